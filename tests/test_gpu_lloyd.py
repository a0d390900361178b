"""Lloyd-Max codebook pools (levels (0, a, 3 - a, 3) per layer, KV head and K|V) against the oracle.

Codes and (scale, zero) bit-exact against the oracle's Lloyd-Max quantiser fed the GPU's own fp32
rotated rows; decode within abs 1e-3 + rel 2e-3 of the oracle's decode with the same codebook;
the library's Lloyd fit equal to the oracle's on the same rotated rows."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from bit_kv_cache_paged_gb300 import Pool
from bit_kv_cache_paged_gb300 import binding as B
from harness import Case, bits_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _codes_bit_exact(c, seq, layer, head, F):
    pos = np.arange(64, F)
    ck, szk, cv, szv = (t.cpu().numpy() for t in c.pool.debug_read_int2(seq, layer, head, 64, F - 64))
    for kv, codes, sz in ((0, ck, szk), (1, cv, szv)):
        raw = c.rows(seq, layer, head, kv, pos)
        rot32 = c.pool.debug_rotate_rows(layer, head, kv, bits_to_dev(raw, (pos.size, 128))).cpu().numpy()
        oc, os_, oz, bad = O.quantize_lloyd_fp32(rot32, c.clip, c.G, c.lloyd_a[layer, head, kv])
        assert not bad.any()
        np.testing.assert_array_equal(codes, O.pack_codes(oc), err_msg=f"codes kv={kv}")
        np.testing.assert_array_equal(sz[..., 0].view(np.uint16), os_.view(np.uint16))
        np.testing.assert_array_equal(sz[..., 1].view(np.uint16), oz.view(np.uint16))


def test_fit_codebook_equals_oracle_fit():
    c = Case(layers=2, Hq=8, Hkv=2, lloyd_a=np.ones((2, 2, 2)))
    for layer, head, kv in ((0, 0, 0), (1, 1, 1), (0, 1, 1)):
        raw = c.rows(1000 + layer, layer, head, kv, np.arange(2048))
        x = bits_to_dev(raw, (2048, 128))
        a_gpu = c.pool.fit_codebook(layer, head, kv, x, iters=50)
        rot32 = c.pool.debug_rotate_rows(layer, head, kv, x).cpu().numpy()
        a_or = O.lloyd_fit(O.normalized_rows(rot32, c.clip, c.G), iters=50)
        assert abs(a_gpu - np.float32(a_or)) <= 1e-6, (a_gpu, a_or)
        assert 1.0 < a_or < 1.45  # rotated rows are bell-shaped: interior levels move inward


@pytest.mark.parametrize("G,absorbed,Hq", [(128, False, 4), (32, False, 4), (128, True, 8), (32, False, 8)])
def test_lloyd_prefill_decode_parity(G, absorbed, Hq):
    a = np.array([[[1.17, 0.82]]], np.float32) if Hq == 4 else np.array([[[1.3, 1.05]]], np.float32)
    c = Case(layers=1, Hq=Hq, Hkv=1, G=G, absorbed=absorbed, lloyd_a=a)
    c.add(0)
    c.step([0], [2045])
    for k in range(3):
        c.step([0], [1])
        c.check_decode(0, k, [0])
    L, F, _ = c.pool.seq_info(0)
    _codes_bit_exact(c, 0, 0, 0, F)


def test_lloyd_ragged_batch_two_layers():
    lengths = [1, 300, 1000, 2048, 4600]
    a = np.array([[[1.1, 1.2], [0.9, 1.0]], [[1.25, 0.75], [1.0, 1.4]]], np.float32)
    c = Case(layers=2, Hq=8, Hkv=2, max_seqs=len(lengths), max_len=5000, lloyd_a=a)
    ids = list(range(len(lengths)))
    for s in ids:
        c.add(s)
    c.step(ids, [L - 1 for L in lengths])
    c.step(ids, [1] * len(ids))
    for layer in range(2):
        c.check_decode(layer, 0, ids)
    _codes_bit_exact(c, ids[-1], 1, 1, c.pool.seq_info(ids[-1])[1])


def test_codebook_a1_equals_uniform_pool():
    """A Lloyd-Max pool at a = 1 stores the same codes and decodes like a uniform pool."""
    u = Case(layers=1, Hq=4, Hkv=1)
    m = Case(layers=1, Hq=4, Hkv=1, lloyd_a=np.ones((1, 1, 2)))
    for c in (u, m):
        c.add(0)
        c.step([0], [3000])
    F = u.pool.seq_info(0)[1]
    for x, y in zip(u.pool.debug_read_int2(0, 0, 0, 64, F - 64), m.pool.debug_read_int2(0, 0, 0, 64, F - 64)):
        assert torch.equal(x, y)
    q = bits_to_dev(u.q_bits(0, [0]), (1, 4, 128))
    ou, om = u.pool.attend(0, q), m.pool.attend(0, q)
    assert torch.allclose(ou, om, atol=2e-5, rtol=1e-5)


def test_set_codebook_rules():
    dev = torch.device("cuda")
    U = torch.eye(128, device=dev)[None, None].contiguous()
    clip = torch.full((1, 1), 0.9, device=dev)
    plain = Pool(1, 4, 1, 2, 1000, 32, U_k=U, U_v=U, clip_k=clip, clip_v=clip)
    with pytest.raises(B.OscarError) as e:
        plain.set_codebook([[[1.0, 1.0]]])  # not a Lloyd-Max pool
    assert e.value.status == B.OSCAR_EINVAL
    lm = Pool(1, 4, 1, 2, 1000, 32, U_k=U, U_v=U, clip_k=clip, clip_v=clip, lloyd_max=True)
    for bad in ([[[0.4, 1.0]]], [[[1.0, 1.5]]], [[[float("nan"), 1.0]]]):
        with pytest.raises(B.OscarError) as e:
            lm.set_codebook(bad)
        assert e.value.status == B.OSCAR_EINVAL
    lm.set_codebook([[[1.2, 0.8]]])
    lm.seq_add(0)
    lm.step_begin([0], [10])
    with pytest.raises(B.OscarError) as e:
        lm.set_codebook([[[1.0, 1.0]]])  # codes already depend on it
    assert e.value.status == B.OSCAR_ESTATE
    plain.close()
    lm.close()


@pytest.mark.parametrize("a", [None, 1.25])
def test_codes_at_exact_decision_thresholds(a):
    """V rows that land exactly on the decision thresholds (absorbed V: R = I; group min 0, max 3,
    clip 1: s = 1, z = 0, u = x): the demote's fast quotient must defer to the exact rule there."""
    dev = torch.device("cuda")
    U = torch.eye(128, device=dev)[None, None].contiguous()
    one = torch.ones((1, 1), device=dev)
    p = Pool(1, 4, 1, 2, 2000, 40, U_k=U, U_v=U, clip_k=one, clip_v=one, v_rot_absorbed=True,
             lloyd_max=a is not None)
    if a is not None:
        p.set_codebook([[[1.0, a]]])
    rng = np.random.default_rng(21)
    n = 700
    ties = np.array([0.5, 1.5, 2.5, 0.625, 2.375, 1.0, 2.0, 0.75, 2.25], np.float32)
    v = rng.choice(ties, size=(n, 128)).astype(np.float32)
    v[:, 0], v[:, 1] = 0.0, 3.0
    k = rng.standard_normal((n, 128)).astype(np.float32)
    tob = lambda x: torch.from_numpy(W.f32_to_bf16_bits(x).view(np.int16)).view(torch.bfloat16).to(dev).view(n, 1, 128)  # noqa: E731
    p.seq_add(0)
    p.step_begin([0], [n])
    p.append_and_demote(0, tob(k), tob(v))
    p.check()
    F = p.seq_info(0)[1]
    _, _, cv, szv = (t.cpu().numpy() for t in p.debug_read_int2(0, 0, 0, 64, F - 64))
    x = W.bf16_bits_to_f32(W.f32_to_bf16_bits(v[64:F]))
    if a is None:
        oc, os_, oz, _ = O.quantize_fp32(x, np.float32(1.0), 128)
    else:
        oc, os_, oz, _ = O.quantize_lloyd_fp32(x, np.float32(1.0), 128, a)
    assert float(os_[0, 0]) == 1.0 and float(oz[0, 0]) == 0.0
    np.testing.assert_array_equal(cv, O.pack_codes(oc))
    np.testing.assert_array_equal(szv[..., 0].view(np.uint16), os_.view(np.uint16))
    p.close()
