"""Parity at the full workload sizes, in the launch configuration the benchmark times.

Each test fills a whole cache on the GPU with the benchmark's fill (device generator + bulk demote),
runs one decode step over every layer (append 1 token per sequence, demote 1, rotate_q, decode,
merge), and checks sampled (sequence, layer, KV head) units against the fp64 oracle one by one:
every query head of the unit within abs 1e-3 + rel 2e-3, and the packed codes and fp16 (scale, zero)
of sampled position ranges bit-exact against the oracle's fp32 quantiser fed the GPU's own rotated
rows. Workloads:
  * Qwen3-8B shape, 36 layers, 32 sequences x 100000 tokens, 32 q / 8 KV heads, group 128;
  * Qwen3-32B shape, 64 layers, 8 sequences x 131072 tokens, 64 q / 8 KV heads, group 128 and 32;
  * ragged serving batch: 64 sequences, lognormal lengths 1K-128K, 26 of them sharing a
    32768-token prefix through shared page-table entries, 36 layers, 32 q / 8 KV heads."""
import numpy as np
import pytest
import torch

import bench
import oracle as O
import workloads as W
from harness import assert_close_decode

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SEED = 0


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _key(share, s, pos):
    """Generator key (sequence id) of a position: shared-prefix positions belong to the owner."""
    if share is not None and s in share[2] and s != share[0] and pos < share[1]:
        return share[0]
    return s


def _rows(masks, share, s, l, h, kv, positions):
    positions = np.asarray(positions, np.int64)
    out = np.zeros((positions.size, 128), np.uint16)
    keys = np.array([_key(share, s, int(p)) for p in positions]) if positions.size else np.zeros(0, int)
    for k in np.unique(keys):
        sel = keys == k
        out[sel] = W.kv_rows_bf16(SEED, int(k), l, h, kv, positions[sel], masks[l, kv, h].astype(bool))
    return out


def _decode_step(pool, wl, lengths, masks, dev):
    """One benchmark-shaped step: every sequence appends the token at its current length."""
    from workloads import device as wd

    B, _, NL, Hq, Hkv, _ = wl
    mdev = torch.from_numpy(masks).to(dev)
    st = torch.cuda.current_stream().cuda_stream
    pool.step_begin(list(range(B)), [1] * B)
    k = torch.empty((B, Hkv, 128), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    q_rot = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    outs = []
    for l in range(NL):
        for s in range(B):
            wd.fill_kv(k[s:s + 1], SEED, s, l, 0, 0, Hkv, int(lengths[s]), 1, mdev[l, 0], st)
            wd.fill_kv(v[s:s + 1], SEED, s, l, 1, 0, Hkv, int(lengths[s]), 1, mdev[l, 1], st)
        qb = np.stack([W.q_rows_bf16(SEED, l, s, np.arange(Hq)) for s in range(B)])
        q = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).to(dev)
        pool.append_and_demote(l, k, v)
        pool.rotate_q(l, q, q_rot)
        part = pool.decode(l, q, q_rot)
        outs.append((qb, pool.merge(l, part).cpu().numpy()))
    pool.check()
    return outs


def _check_unit(pool, wl, U, masks, share, outs, s, l, h, demote_ranges):
    B, _, NL, Hq, Hkv, G = wl
    hg = Hq // Hkv
    L, F, _ = pool.seq_info(s)
    ck, szk, cv, szv = (t.cpu().numpy() for t in pool.debug_read_int2(s, l, h, 64, F - 64))
    pos_b = np.r_[0:min(64, L), F:L]
    kb = W.bf16_bits_to_f32(_rows(masks, share, s, l, h, 0, pos_b))
    vb = W.bf16_bits_to_f32(_rows(masks, share, s, l, h, 1, pos_b))
    # the BF16 zones hold the generator rows
    for p0, n in ((0, min(64, L)), (F, L - F)):
        kd, vd = (t.view(torch.int16).cpu().numpy().view(np.uint16) for t in pool.debug_read_bf16(s, l, h, p0, n))
        np.testing.assert_array_equal(kd, _rows(masks, share, s, l, h, 0, np.arange(p0, p0 + n)))
        np.testing.assert_array_equal(vd, _rows(masks, share, s, l, h, 1, np.arange(p0, p0 + n)))
    qb, out = outs[l]
    qf = W.bf16_bits_to_f32(qb[s, h * hg:(h + 1) * hg])
    ref, _ = O.decode_reference(qf, kb, vb, O.unpack_codes(ck), szk[..., 0], szk[..., 1], O.unpack_codes(cv),
                                szv[..., 0], szv[..., 1], U[0, l, h], U[1, l, h], G)
    assert_close_decode(out[s, h * hg:(h + 1) * hg], ref, f"seq {s} layer {l} kv head {h}")
    # bit-exact demote on sampled position ranges
    for a, b in demote_ranges(F):
        pos = np.arange(a, b)
        for kv, codes, sz in ((0, ck, szk), (1, cv, szv)):
            raw = _rows(masks, share, s, l, h, kv, pos)
            x = torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16).cuda()
            rot = pool.debug_rotate_rows(l, h, kv, x).cpu().numpy()
            oc, os_, oz, bad = O.quantize_fp32(rot, np.float32(0.9), G)
            assert not bad.any()
            np.testing.assert_array_equal(codes[a - 64:b - 64], O.pack_codes(oc), err_msg=f"codes kv={kv}")
            np.testing.assert_array_equal(sz[a - 64:b - 64, :, 0].view(np.uint16), os_.view(np.uint16))
            np.testing.assert_array_equal(sz[a - 64:b - 64, :, 1].view(np.uint16), oz.view(np.uint16))


def _run(wl, lengths, share, units):
    dev = torch.device("cuda")
    pool, U, masks = bench.build_pool(wl, SEED, 4, dev, lengths)
    try:
        bench.fill_cache(pool, wl, lengths, masks, SEED, dev, share)
        outs = _decode_step(pool, wl, lengths, masks, dev)
        for s, l, h in units:
            # first two pages, and the newest INT2 tokens (the last one demoted by the decode step)
            _check_unit(pool, wl, U, masks, share, outs, s, l, h,
                        lambda F: [(64, min(F, 64 + 128)), (max(64, F - 96), F)])
    finally:
        pool.close()
        del pool
        torch.cuda.empty_cache()


def _units(wl, n, rng, extra=()):
    B, _, NL, _, Hkv, _ = wl
    u = [(0, 0, 0), (B - 1, NL - 1, Hkv - 1)] + list(extra)
    u += [(int(rng.integers(B)), int(rng.integers(NL)), int(rng.integers(Hkv))) for _ in range(n)]
    return u


def test_qwen3_8b_b32_100k_sampled_parity():
    wl = bench.WORKLOADS["qwen3_8b_b32_100k"]
    lengths = np.full(wl[0], wl[1] - 1, np.int64)  # the decode step appends token 99999
    _run(wl, lengths, None, _units(wl, 6, np.random.default_rng(1)))


@pytest.mark.parametrize("name", ["qwen3_32b_b8_128k", "qwen3_32b_b8_128k_g32"])
def test_qwen3_32b_b8_128k_sampled_parity(name):
    wl = bench.WORKLOADS[name]
    lengths = np.full(wl[0], wl[1] - 1, np.int64)
    _run(wl, lengths, None, _units(wl, 5, np.random.default_rng(2)))


def test_ragged_b64_shared_prefix_sampled_parity():
    lengths, sharers = W.config4_lengths(SEED)
    wl = (64, int(lengths.max()), 36, 32, 8, 128)
    share = (int(sharers[0]), 32768, set(int(x) for x in sharers))
    lengths = lengths - 1  # the decode step appends each sequence's last token
    # the prefix owner, two sharers, the shortest and the longest sequence, and random ones
    extra = [(int(sharers[0]), 3, 2), (int(sharers[1]), 17, 5), (int(sharers[-1]), 35, 7),
             (int(np.argmin(lengths)), 10, 1), (int(np.argmax(lengths)), 20, 6)]
    _run(wl, lengths, share, _units(wl, 4, np.random.default_rng(3), extra))
