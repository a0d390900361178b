"""BF16-only paged cache decode (the comparison cache) against the oracle's fp64 softmax attention.

Pages are handed out in a shuffled order so the page table is exercised; lengths cover an empty
tail page, exact page multiples, several 32-page chunks and a ragged tail."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from bit_kv_cache_paged_gb300 import binding as B
from harness import assert_close_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 2)])
def test_bf16_paged_decode_vs_oracle(Hq, Hkv):
    seed, layer = 0, 0
    lengths = np.array([1, 63, 64, 65, 2048, 2049, 5000], np.int32)
    n = lengths.size
    max_len = int(lengths.max())
    maxp = (max_len + 63) // 64
    n_pages = int(sum((L + 63) // 64 for L in lengths))
    rng = np.random.default_rng(5)
    perm = rng.permutation(n_pages).astype(np.int32)
    pt = np.full((n, maxp), -1, np.int32)
    k_off = 0
    for i, L in enumerate(lengths):
        npg = (int(L) + 63) // 64
        pt[i, :npg] = perm[k_off:k_off + npg]
        k_off += npg
    dev = torch.device("cuda")
    st = torch.cuda.current_stream().cuda_stream
    kp = torch.zeros((n_pages, Hkv, 64, 128), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pt_d = torch.from_numpy(pt).to(dev)
    masks = {(h, kv): W.outlier_mask_bernoulli(seed, layer, h, kv).astype(bool) for h in range(Hkv) for kv in (0, 1)}
    rows = {}
    for i, L in enumerate(lengths):
        pos = np.arange(int(L))
        for kv, dst in ((0, kp), (1, vp)):
            r = np.stack([W.kv_rows_bf16(seed, i, layer, h, kv, pos, masks[h, kv]) for h in range(Hkv)], axis=1)
            rows[i, kv] = r
            rd = torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).to(dev)
            B.oscar_bf16_pack(rd, int(L), 0, Hkv, pt_d[i], n_pages, dst, err, st)
    qb = np.stack([W.q_rows_bf16(seed, 0, i, np.arange(Hq)) for i in range(n)])
    q = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).to(dev)
    nb = B.oscar_bf16_partials_bytes(Hq, Hkv, n, max_len)
    part = torch.empty(nb, dtype=torch.uint8, device=dev)
    out = torch.full((n, Hq, 128), float("nan"), device=dev)
    L_d = torch.from_numpy(lengths).to(dev)
    for rep in range(2):  # the second call reuses the scratch
        B.oscar_bf16_decode(Hq, Hkv, n, max_len, kp, vp, n_pages, pt_d, maxp, L_d, q, part, nb, out, err, st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.cpu().numpy()
        hg = Hq // Hkv
        for i in range(n):
            for h in range(Hkv):
                K = W.bf16_bits_to_f32(rows[i, 0][:, h])
                V = W.bf16_bits_to_f32(rows[i, 1][:, h])
                qf = W.bf16_bits_to_f32(qb[i, h * hg:(h + 1) * hg])
                ref, _ = O.attention(qf, K, V)
                assert_close_decode(got[i, h * hg:(h + 1) * hg], ref, f"seq {i} head {h}")
    # an out-of-range page id is reported, not followed
    pt_bad = pt.copy()
    pt_bad[4, 0] = n_pages + 7
    B.oscar_bf16_decode(Hq, Hkv, n, max_len, kp, vp, n_pages, torch.from_numpy(pt_bad).to(dev), maxp, L_d, q, part,
                        nb, out, err, st)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DEVERR_PAGE
