"""GPU parity of liboscar (called through its C ABI) against the CPU oracle.

Bars: packed codes and fp16 (scale, zero) bit-exact against the oracle's fp32 quantiser fed the
GPU's own fp32 rotated rows; rotated rows within 1e-5 * |x| of the fp64 rotation; decode output
within abs 1e-3 + rel 2e-3 of the fp64 oracle on the same packed cache."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from harness import Case, assert_close_decode, bits_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def test_device_generator_matches_host():
    from workloads import device as wd
    m = torch.from_numpy(np.stack([W.outlier_mask_bernoulli(0, 3, h, 1) for h in range(8)]).astype(np.uint8)).cuda()
    out = torch.empty((300, 8, 128), dtype=torch.bfloat16, device="cuda")
    wd.fill_kv(out, 0, 5, 3, 1, 0, 8, 70000, 300, m, torch.cuda.current_stream().cuda_stream)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    for h in range(8):
        want = W.kv_rows_bf16(0, 5, 3, h, 1, np.arange(70000, 70300), m[h].cpu().numpy().astype(bool))
        np.testing.assert_array_equal(got[:, h], want)


@pytest.mark.parametrize("absorbed", [False, True])
def test_rotation_rows_vs_fp64(absorbed):
    c = Case(layers=2, Hq=8, Hkv=2, absorbed=absorbed)
    rng = np.random.default_rng(0)
    x = W.f32_to_bf16_bits((rng.standard_normal((200, 128)) * np.where(rng.random(128) < 0.05, 20, 1)).astype(np.float32))
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    for layer in range(2):
        for h in range(2):
            for kv in range(2):
                got = c.pool.debug_rotate_rows(layer, h, kv, bits_to_dev(x, (200, 128))).cpu().numpy()
                if kv == 1 and absorbed:
                    np.testing.assert_array_equal(got, xf.astype(np.float32))
                    continue
                ref = xf @ O.rotation_matrix(c.U[kv, layer, h])
                err = np.abs(got - ref).max(axis=1)
                assert np.all(err <= 1e-5 * np.linalg.norm(xf, axis=1)), err.max()


def _demote_bit_exact(c, seq, layer, head, F):
    """Codes and (s, z) of INT2 positions [64, F): GPU vs oracle quantiser on GPU rotated rows."""
    pos = np.arange(64, F)
    ck, szk, cv, szv = (t.cpu().numpy() for t in c.pool.debug_read_int2(seq, layer, head, 64, F - 64))
    for kv, codes, sz in ((0, ck, szk), (1, cv, szv)):
        raw = c.rows(seq, layer, head, kv, pos)
        rot32 = c.pool.debug_rotate_rows(layer, head, kv, bits_to_dev(raw, (pos.size, 128))).cpu().numpy()
        oc, os_, oz, bad = O.quantize_fp32(rot32, c.clip, c.G)
        assert not bad.any()
        np.testing.assert_array_equal(codes, O.pack_codes(oc), err_msg=f"codes kv={kv}")
        np.testing.assert_array_equal(sz[..., 0].view(np.uint16), os_.view(np.uint16), err_msg="scale")
        np.testing.assert_array_equal(sz[..., 1].view(np.uint16), oz.view(np.uint16), err_msg="zero")
        # fully independent encoding (fp64 rotation rounded to fp32): agrees except at rounding ties
        enc = O.encode_rows(W.bf16_bits_to_f32(raw), c.U[kv, layer, head], c.clip, c.G,
                            rotate=not (kv == 1 and c.absorbed))
        mism = (enc["codes"] != oc).mean()
        assert mism < 1e-3, mism


@pytest.mark.parametrize("G,absorbed,Hq", [(128, False, 4), (32, False, 4), (128, True, 4), (128, False, 8),
                                           (32, True, 8)])
def test_tiny_prefill_then_decode_steps(G, absorbed, Hq):
    """configs[0]-shaped: 1 seq, 2048 tokens = 64 sink + 1728 INT2 + 256 recent; then decode steps
    (append 1 + demote 1 from the recent ring) with parity after each."""
    c = Case(layers=1, Hq=Hq, Hkv=1, G=G, absorbed=absorbed)
    c.add(0)
    c.step([0], [2045])
    for k in range(3):
        c.step([0], [1])
        L, F, _ = c.pool.seq_info(0)
        assert L == 2046 + k and F == L - 256
        c.check_decode(0, k, [0])
    assert (L, F) == (2048, 1792)
    _demote_bit_exact(c, 0, 0, 0, F)
    # BF16 zones hold the generator rows (sink + recent ring)
    for p0, n in ((0, 64), (F, L - F)):
        k, v = (t.view(torch.int16).cpu().numpy().view(np.uint16) for t in c.pool.debug_read_bf16(0, 0, 0, p0, n))
        np.testing.assert_array_equal(k, c.rows(0, 0, 0, 0, np.arange(p0, p0 + n)))
        np.testing.assert_array_equal(v, c.rows(0, 0, 0, 1, np.arange(p0, p0 + n)))


def test_rotate_q_vs_oracle():
    c = Case(layers=2, Hq=16, Hkv=2)
    for s in range(3):
        c.add(s)
    c.step([0, 1, 2], [10, 20, 30])
    qb = c.q_bits(0, [0, 1, 2])
    q = bits_to_dev(qb, (3, 16, 128))
    for layer in range(2):
        got = c.pool.rotate_q(layer, q).cpu().numpy()
        for h in range(16):
            ref = W.bf16_bits_to_f32(qb[:, h]).astype(np.float64) @ O.rotation_matrix(c.U[0, layer, h // 8])
            assert np.abs(got[:, h] - ref).max() <= 1e-5 * np.abs(ref).max() * 11.3


@pytest.mark.parametrize("G", [128, 32])
def test_ragged_batch_many_lengths(G):
    """Ragged batch across zone boundaries, tiles and partial tail pages, 2 layers, 2 KV heads."""
    lengths = [1, 63, 64, 65, 300, 320, 321, 385, 1000, 2048, 3001, 4600]
    c = Case(layers=2, Hq=8, Hkv=2, G=G, max_seqs=len(lengths), max_len=5000)
    ids = list(range(len(lengths)))
    for s in ids:
        c.add(s)
    c.step(ids, [L - 1 for L in lengths])
    c.step(ids, [1] * len(ids))
    for layer in range(2):
        c.check_decode(layer, 0, ids)
    # every sequence's history: the prefill's tiles straddle sequences (per-thread row copies) or
    # lie inside one sequence's new tokens (tensor copies); both must give the spec's codes
    for s in ids:
        F = c.pool.seq_info(s)[1]
        if F > 64:
            _demote_bit_exact(c, s, 1, 1, F)


def test_batch_order_is_step_order():
    """Batch index i of q/out follows the seq_ids order passed to step_begin, not the ids."""
    c = Case(layers=1, Hq=4, Hkv=1, max_seqs=3, max_len=3000)
    for s in (2, 0, 1):
        c.add(s)
    c.step([2, 0, 1], [2500, 700, 1300])
    c.step([1, 2, 0], [1, 1, 1])
    c.check_decode(0, 0, [1, 2, 0])


def test_prefix_sharing_decode():
    """Sequences sharing a prefix through page-table entries decode like independent copies."""
    c = Case(layers=1, Hq=8, Hkv=2, max_seqs=4, max_len=6000)
    c.add(0)
    c.step([0], [64 + 64 * 40 + 256 + 100])
    c.add(1, 0, 64 + 64 * 40)
    c.add(2, 0, 64 + 64 * 20)
    c.step([1, 2], [700, 300])
    c.step([0, 1, 2], [1, 1, 1])
    c.check_decode(0, 0, [0, 1, 2])
    st = c.pool.stats()
    own = [c.pool.seq_info(s)[2] for s in (0, 1, 2)]
    assert st["int2_pages_used"] == own[0] + (own[1] - 40) + (own[2] - 20)


def test_multistep_ring_wraparound():
    """Many single-token steps: the recent ring wraps and every demoted token comes from the ring."""
    c = Case(layers=1, Hq=4, Hkv=1, G=32, max_len=2000)
    c.add(0)
    c.step([0], [300])
    for k in range(300):
        c.step([0], [1])
    L, F, _ = c.pool.seq_info(0)
    assert (L, F) == (600, 344)
    c.check_decode(0, 0, [0])
    _demote_bit_exact(c, 0, 0, 0, F)


def test_chunked_prefill_demotes_ring_and_new_rows():
    """A second prefill chunk demotes the previous chunk's recent window (rows from the BF16 ring,
    not page-aligned) and its own first tokens (rows from k_new / v_new) in one bulk launch."""
    for G in (128, 32):
        c = Case(layers=1, Hq=4, Hkv=1, G=G, max_len=3000)
        c.add(0)
        c.step([0], [1000])  # history [64, 744)
        c.step([0], [700])   # demotes [744, 1444): 256 ring rows, then 444 new rows
        L, F, _ = c.pool.seq_info(0)
        assert (L, F) == (1700, 1444)
        c.check_decode(0, 0, [0])
        _demote_bit_exact(c, 0, 0, 0, F)


def test_decode_step_of_many_sequences_uses_the_bulk_demote():
    """A decode step of 40 sequences demotes 40 rows per (KV head, K|V), more than the four-lane
    form takes (32): the bulk form then demotes one ring row per sequence, every tile spanning
    sequences. The codes of the step's demoted positions match the spec."""
    n = 40
    c = Case(layers=1, Hq=4, Hkv=1, max_seqs=n, max_len=1200)
    ids = list(range(n))
    for s_ in ids:
        c.add(s_)
    c.step(ids, [400 + 3 * s_ for s_ in ids])  # every sequence past its recent window
    c.step(ids, [1] * n)                        # one demoted row each, from the ring
    c.check_decode(0, 0, ids)
    for s_ in (0, 17, n - 1):
        _demote_bit_exact(c, s_, 0, 0, c.pool.seq_info(s_)[1])


def test_device_error_word_for_non_finite_input():
    c = Case(layers=1, Hq=4, Hkv=1)
    c.add(0)
    c.pool.step_begin([0], [400])
    k = torch.zeros((400, 1, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((400, 1, 128), dtype=torch.bfloat16, device="cuda")
    k[100, 0, 5] = float("nan")
    c.pool.append_and_demote(0, k, v)
    from bit_kv_cache_paged_gb300.binding import OscarError, DEVERR_INPUT
    with pytest.raises(OscarError) as e:
        c.pool.check()
    assert e.value.detail & DEVERR_INPUT
    c.pool.check()  # cleared


def test_qwen3_8b_layer_full_parity():
    """Qwen3-8B-shaped layer: batch 1, 32 q / 8 KV heads, context 32768 (32448 INT2 tokens)."""
    c = Case(layers=1, Hq=32, Hkv=8, outliers="bernoulli", max_seqs=1, max_len=33000)
    c.add(0)
    c.step([0], [32767])
    c.step([0], [1])
    assert c.pool.seq_info(0)[:2] == (32768, 32512)
    c.check_decode(0, 0, [0])
    _demote_bit_exact(c, 0, 0, 5, 32512)


def test_bounded_wait_timeout_is_reported_not_hung():
    """A kernel waiting on an mbarrier that nothing completes gives up (~0.5 s), sets the timeout
    bit of the device error word and returns; the context stays usable."""
    from bit_kv_cache_paged_gb300 import binding as B
    c = Case(layers=1, Hq=4, Hkv=1)
    B.oscar_debug_timeout_selftest(c.pool.handle, torch.cuda.current_stream().cuda_stream)
    st, detail = B.oscar_check(c.pool.handle, torch.cuda.current_stream().cuda_stream)
    assert st == B.OSCAR_ETIMEOUT and detail & B.DEVERR_TIMEOUT
    assert B.oscar_check(c.pool.handle, torch.cuda.current_stream().cuda_stream) == (B.OSCAR_OK, 0)
    c.add(0)  # the pool still works afterwards
    c.step([0], [500])
    c.check_decode(0, 0, [0])
