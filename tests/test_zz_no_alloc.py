"""oscar_decode_merge_noalloc: decode + merge with the partials in liboscar's own device array.

The file name makes pytest collect it last, so its GPU tests run both on a fresh process (alone)
and after every other test has used the device. The GPU tests call the entry point through the C
ABI and compare it with oscar_decode + oscar_merge on the same step."""
import re

import numpy as np
import pytest
import torch

import workloads as W
from bit_kv_cache_paged_gb300 import Pool
from bit_kv_cache_paged_gb300 import binding as B
from harness import Case, assert_close_decode, bits_to_dev


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_header_limit_matches_binding():
    import os
    text = open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "oscar.h")).read()
    m = re.search(r"#define OSCAR_NOALLOC_PARTIALS_MAX_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == B.NOALLOC_PARTIALS_MAX_BYTES


def test_host_only_pool_is_rejected_without_cuda():
    """Argument and state checks come before any CUDA call (host-only pool, no GPU needed)."""
    p = Pool(1, 4, 1, max_seqs=2, max_seq_len=1000, max_int2_pages=32, host_only=True)
    p.seq_add(0)
    with pytest.raises(B.OscarError) as e:
        B.oscar_decode_merge_noalloc(p.handle, 0, 1, 16, 16, 16, None)
    assert e.value.status == B.OSCAR_ESTATE
    p.step_begin([0], [500])
    for layer, n in ((0, 1), (1, 1), (0, 2)):
        with pytest.raises(B.OscarError) as e:
            B.oscar_decode_merge_noalloc(p.handle, layer, n, 16, 16, 16, None)
        assert e.value.status == B.OSCAR_EINVAL
    p.close()


@pytest.fixture(scope="module")
def built():
    import __graft_entry__ as g
    g.build()


def _reference_and_noalloc(c, layers, step, ids, launches_per_layer=3):
    """Existing path for every layer first, then the no-alloc entry point for the same layers
    called back to back (the array is reused between the calls)."""
    q = bits_to_dev(c.q_bits(step, ids), (len(ids), c.Hq, 128))
    q_rot = [c.pool.rotate_q(l, q) for l in layers]
    ref = [c.pool.merge(l, c.pool.decode(l, q, q_rot[k])).clone() for k, l in enumerate(layers)]
    got = [torch.full_like(r, float("nan")) for r in ref]
    n0 = c.pool.launch_count()
    for k, l in enumerate(layers):
        B.oscar_decode_merge_noalloc(c.pool.handle, l, len(ids), q, q_rot[k], got[k], _stream())
    torch.cuda.synchronize()
    c.pool.check()
    assert c.pool.launch_count() - n0 == launches_per_layer * len(layers)
    return q, ref, got


def _check_against_oracle(c, out, step, ids, layer):
    qb = c.q_bits(step, ids)
    for i, s in enumerate(ids):
        for h in range(c.Hkv):
            qf = W.bf16_bits_to_f32(qb[i, h * c.hg:(h + 1) * c.hg])
            want, _ = c.oracle_pair(s, layer, h, qf)
            assert_close_decode(out[i, h * c.hg:(h + 1) * c.hg], want, f"seq {s} head {h}")


@pytest.mark.gpu
def test_noalloc_equals_decode_merge_two_calls_in_a_row(built):
    lengths = [1, 300, 1000, 2048, 4100]
    ids = list(range(len(lengths)))
    c = Case(layers=2, Hq=8, Hkv=2, max_seqs=len(lengths), max_len=5000)
    for s in ids:
        c.add(s)
    c.step(ids, [L - 1 for L in lengths])
    c.step(ids, [1] * len(ids))
    for step in (0, 1):
        if step:
            c.step(ids, [1] * len(ids))
        _, ref, got = _reference_and_noalloc(c, [0, 1], step, ids)
        for r, g in zip(ref, got):
            assert torch.equal(r, g)  # same kernels on the same inputs: bit-identical
    # and against the fp64 oracle, for the last call
    qb = c.q_bits(1, ids)
    out = got[1].cpu().numpy()
    for i, s in enumerate(ids):
        for h in range(c.Hkv):
            qf = W.bf16_bits_to_f32(qb[i, h * c.hg:(h + 1) * c.hg])
            want, _ = c.oracle_pair(s, 1, h, qf)
            assert_close_decode(out[i, h * c.hg:(h + 1) * c.hg], want, f"seq {s} head {h}")


@pytest.mark.gpu
def test_noalloc_eight_query_heads_per_kv_head(built):
    """A pool with 8 query heads per KV head launches other kernel instances than the test above;
    their first call loads them, and two calls in a row match oscar_decode + oscar_merge."""
    lengths = [700, 2100, 333]
    ids = list(range(len(lengths)))
    c = Case(layers=1, Hq=16, Hkv=2, max_seqs=len(lengths), max_len=3000)
    for s in ids:
        c.add(s)
    c.step(ids, lengths)
    for step in (0, 1):
        if step:
            c.step(ids, [1] * len(ids))
        _, ref, got = _reference_and_noalloc(c, [0], step, ids)
        assert torch.equal(ref[0], got[0])
    _check_against_oracle(c, got[0].cpu().numpy(), 1, ids, 0)


@pytest.mark.gpu
def test_noalloc_step_without_int2_history(built):
    """Every sequence shorter than 64 + 256 tokens: no INT2 unit, so only the BF16 kernel and the
    merge run (two launches per call), and the merge reads no INT2 slot."""
    lengths = [1, 64, 200, 319]
    ids = list(range(len(lengths)))
    c = Case(layers=2, Hq=8, Hkv=2, max_seqs=len(lengths), max_len=1000)
    for s in ids:
        c.add(s)
    c.step(ids, lengths)
    assert all(c.pool.seq_info(s)[1] == 64 for s in ids)
    assert c.pool.partials_bytes() > 0
    _, ref, got = _reference_and_noalloc(c, [0, 1], 0, ids, launches_per_layer=2)
    for r, g in zip(ref, got):
        assert torch.equal(r, g)
    _check_against_oracle(c, got[1].cpu().numpy(), 0, ids, 1)


@pytest.mark.gpu
def test_noalloc_rejects_partials_above_limit(built):
    """Batch 200 x 8 KV heads at 8 query heads per KV head needs more than the fixed array: the
    call fails with OSCAR_EINVAL and launches nothing."""
    dev = torch.device("cuda")
    Hq, Hkv, n = 64, 8, 200
    U = torch.eye(128, device=dev).expand(1, Hkv, 128, 128).contiguous()
    clip = torch.full((1, Hkv), 0.9, device=dev)
    p = Pool(1, Hq, Hkv, max_seqs=n, max_seq_len=1200, max_int2_pages=n * 19, U_k=U, U_v=U.clone(),
             clip_k=clip, clip_v=clip.clone())
    ids = list(range(n))
    for s in ids:
        p.seq_add(s)
    p.step_begin(ids, [1000] * n)
    assert p.partials_bytes() > B.NOALLOC_PARTIALS_MAX_BYTES
    q = torch.zeros((n, Hq, 128), dtype=torch.bfloat16, device=dev)
    q_rot = torch.zeros((n, Hq, 128), dtype=torch.float32, device=dev)
    out = torch.full((n, Hq, 128), 7.0, device=dev)
    n0 = p.launch_count()
    with pytest.raises(B.OscarError) as e:
        B.oscar_decode_merge_noalloc(p.handle, 0, n, q, q_rot, out, _stream())
    assert e.value.status == B.OSCAR_EINVAL
    assert p.launch_count() == n0
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    p.close()
