"""Pins of the CPU oracle against facts that do not come from the oracle itself:
closed forms, independent constructions, invariants, brute force on tiny inputs,
and the numbers the source pages print (tests/golden/paper_numbers.json)."""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "paper_numbers.json")


def sylvester_recursive(d):
    """Independent construction: H_1 = [1], H_2n = [[H, H], [H, -H]] (unnormalised)."""
    H = np.array([[1.0]])
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


# ---------------------------------------------------------------- P1: Hadamard
def test_hadamard_matches_recursive_construction():
    for d in (2, 8, 128):
        np.testing.assert_array_equal(O.hadamard(d) * math.sqrt(d), sylvester_recursive(d))


def test_hadamard_orthonormal_and_symmetric():
    H = O.hadamard(128)
    np.testing.assert_allclose(H @ H.T, np.eye(128), atol=1e-12)
    np.testing.assert_array_equal(H, H.T)
    assert np.allclose(H[0], 1 / math.sqrt(128))
    assert np.allclose(H[1], [(-1) ** j / math.sqrt(128) for j in range(128)])


# ---------------------------------------------------------------- P2: bit reversal
def test_bitrev_values_and_involution():
    assert O.bitrev(1, 7) == 64
    assert O.bitrev(3, 7) == 96
    assert O.bitrev(0b0000101, 7) == 0b1010000
    perm = [O.bitrev(i, 7) for i in range(128)]
    assert sorted(perm) == list(range(128))
    assert all(O.bitrev(O.bitrev(i, 7), 7) == i for i in range(128))


def test_bitrev_matrix_semantics():
    P = O.bitrev_matrix(128)
    np.testing.assert_array_equal(P @ P, np.eye(128))
    y = np.arange(128, dtype=np.float64)
    yp = y @ P
    assert all(yp[j] == O.bitrev(j, 7) for j in range(128))


# ---------------------------------------------------------------- P3: U and R
@pytest.fixture(scope="module")
def basis():
    return W.synthetic_basis(0, 0, 0, 0)


def test_synthetic_basis_is_eigenbasis(basis):
    U, C, lam = basis
    U64 = U.astype(np.float64)
    np.testing.assert_allclose(U64.T @ U64, np.eye(128), atol=2e-6)
    np.testing.assert_allclose(C @ U64, U64 * lam, atol=2e-6 * lam[0])
    assert np.all(np.diff(lam) <= 0)
    # spectrum 1/i within the sampling error of 8192 samples
    assert abs(np.trace(C) / sum(1 / i for i in range(1, 129)) - 1) < 0.05
    assert 1.5 < lam[0] / lam[1] < 2.7
    # sign convention: the largest-magnitude entry of each column is positive
    idx = np.argmax(np.abs(U), axis=0)
    assert np.all(U[idx, np.arange(128)] > 0)


def test_rotation_orthogonal(basis):
    R = O.rotation_matrix(basis[0])
    np.testing.assert_allclose(R @ R.T, np.eye(128), atol=2e-6)


def test_rotation_closed_form_on_basis_vectors(basis):
    """Row k of U^T rotates to H[k, bitrev(j)] at position j: pins the order U, then H, then P
    and the row-vector convention (a transposed U or a swapped order fails this)."""
    U = basis[0]
    R = O.rotation_matrix(U)
    for k in (0, 1, 5, 77, 127):
        x = U[:, k].astype(np.float64)
        got = x @ R
        want = np.array([(-1) ** bin(k & O.bitrev(j, 7)).count("1") for j in range(128)]) / math.sqrt(128)
        np.testing.assert_allclose(got, want, atol=2e-6)


# ---------------------------------------------------------------- P4: rotation invariance
def test_rotation_preserves_dot_products(basis):
    R = O.rotation_matrix(basis[0])
    rng = np.random.default_rng(1)
    q = rng.standard_normal((4, 128))
    k = rng.standard_normal((9, 128))
    # R is exactly orthogonal only up to the fp32 rounding of U: compare with R's own Gram
    np.testing.assert_allclose((q @ R) @ (k @ R).T, q @ (R @ R.T) @ k.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose((q @ R) @ (k @ R).T, q @ k.T, rtol=0, atol=1e-4)
    Rh = O.hadamard() @ O.bitrev_matrix()  # exactly orthogonal part
    np.testing.assert_allclose((q @ Rh) @ (k @ Rh).T, q @ k.T, rtol=1e-9, atol=1e-9)


# ---------------------------------------------------------------- P5: quantiser
def test_half_rn_matches_struct_rounding():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(2000).astype(np.float32) * 10,
                         np.float32([65504.0, 6.1035156e-05, 5.96e-08, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11,
                                     2049.0, 2051.0, -0.0, 1e-9, 65519.0])])
    got = O.half_rn(xs).view(np.uint16)
    want = np.array([O.fp16_bits_python(float(x)) for x in xs], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


def test_pack_layout_and_roundtrip():
    codes = np.zeros(128, dtype=np.uint8)
    codes[:4] = [1, 2, 3, 0]
    codes[4:8] = [3, 3, 3, 3]
    p = O.pack_codes(codes)
    assert p.shape == (32,)
    assert p[0] == 1 | 2 << 2 | 3 << 4 and p[1] == 0xFF
    rng = np.random.default_rng(3)
    c = rng.integers(0, 4, size=(50, 128), dtype=np.uint8)
    np.testing.assert_array_equal(O.unpack_codes(O.pack_codes(c)), c)


@pytest.mark.parametrize("G", [128, 32])
def test_quantiser_grid_exact_is_lossless(G):
    rng = np.random.default_rng(4)
    s = np.float32(0.25)
    z = np.float32(-0.5)
    k = rng.integers(0, 4, size=(20, 128))
    k[:, ::G] = 0  # both ends present in every group
    k[:, 1::G] = 3
    x = (z + k * s).astype(np.float32)
    codes, s16, z16, bad = O.quantize_fp32(x, np.float32(1.0), G)
    assert not bad.any()
    np.testing.assert_array_equal(codes, k)
    np.testing.assert_array_equal(s16.astype(np.float32), s)
    np.testing.assert_array_equal(O.dequantize(codes, s16, z16, G), x.astype(np.float64))


@pytest.mark.parametrize("G,clip", [(128, 0.9), (32, 0.9), (128, 1.0)])
def test_quantiser_nearest_level_brute_force(G, clip):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((400, 128)) * np.where(rng.random(128) < 0.05, 20, 1)).astype(np.float32)
    codes, s16, z16, bad = O.quantize_fp32(x, np.float32(clip), G)
    assert not bad.any()
    assert codes.max() <= 3
    sf = np.repeat(s16.astype(np.float64), G, axis=-1)
    zf = np.repeat(z16.astype(np.float64), G, axis=-1)
    levels = zf[..., None] + sf[..., None] * np.arange(4)
    dist = np.abs(x.astype(np.float64)[..., None] - levels)
    best = np.argmin(dist, axis=-1)
    mism = best != codes
    # the only allowed disagreements are (near-)ties between two levels, where fp32
    # subtraction + division may round either way
    if mism.any():
        t = (x.astype(np.float64) - zf) / sf
        frac = np.abs(t - np.floor(t) - 0.5)
        assert np.all(frac[mism] < 1e-5)
    assert mism.sum() <= 2
    # error bound: inside the clipped range the error is at most half a step
    xhat = O.dequantize(codes, s16, z16, G)
    xc = np.clip(x.astype(np.float64), zf, zf + 3 * sf)
    assert np.all(np.abs(xhat - xc) <= sf / 2 * (1 + 1e-5) + 1e-12)


def test_quantiser_clip_saturates_and_ends_map():
    x = np.linspace(-2, 3, 128, dtype=np.float32)
    codes, s16, z16, _ = O.quantize_fp32(x, np.float32(0.9), 128)
    assert codes[0] == 0 and codes[-1] == 3
    assert np.float32(z16) == O.half_rn(np.float32(0.9) * np.float32(-2.0))
    codes1, _, _, _ = O.quantize_fp32(x, np.float32(1.0), 128)
    assert codes1[0] == 0 and codes1[-1] == 3


def test_quantiser_constant_group_and_overflow():
    x = np.full((1, 128), 0.75, dtype=np.float32)
    codes, s16, z16, bad = O.quantize_fp32(x, np.float32(0.9), 128)
    assert not bad.any() and np.all(codes == 0) and s16[0, 0] == 0
    assert z16[0, 0] == O.half_rn(np.float32(0.9) * np.float32(0.75))
    y = np.zeros((1, 128), dtype=np.float32)
    y[0, 0] = 3e5
    _, _, _, bad = O.quantize_fp32(y, np.float32(0.9), 128)
    assert bad.all()


def test_quantiser_uses_fp16_rounded_scale():
    # s32 = 1/3 * 3 * a is not fp16-exact; codes must be computed with the fp16 value
    x = np.zeros(128, dtype=np.float32)
    x[0], x[1] = 0.0, np.float32(1.0009766)  # max just above 1
    x[2] = np.float32(0.50048828)            # close to the 1.5-step midpoint
    codes, s16, z16, _ = O.quantize_fp32(x, np.float32(1.0), 128)
    sf = np.float32(s16[0])
    t = np.float32(np.float32(x[2] - np.float32(z16[0])) / sf)
    assert codes[2] == int(np.clip(np.rint(t), 0, 3))


# ---------------------------------------------------------------- P6: merge
@pytest.mark.parametrize("chunks", [1, 2, 7, 64])
def test_segment_merge_equals_one_pass(chunks):
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 128))
    K = rng.standard_normal((320, 128)) * 2
    V = rng.standard_normal((320, 128))
    o_ref, lse_ref = O.attention(q, K, V)
    cuts = np.linspace(0, 320, chunks + 1).astype(int)
    parts = [O.attention(q, K[a:b], V[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = O.merge_segments(parts)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12)


def test_merge_empty_segment_is_identity():
    rng = np.random.default_rng(7)
    q, K, V = rng.standard_normal((2, 128)), rng.standard_normal((5, 128)), rng.standard_normal((5, 128))
    part = O.attention(q, K, V)
    empty = O.attention(q, K[:0], V[:0])
    assert np.all(np.isneginf(empty[1]))
    o, lse = O.merge_segments([empty, part, empty])
    np.testing.assert_allclose(o, part[0], rtol=1e-14)
    np.testing.assert_allclose(lse, part[1], rtol=1e-14)


# ---------------------------------------------------------------- P7: attention
def test_attention_brute_force_logsumexp():
    rng = np.random.default_rng(8)
    q, K, V = rng.standard_normal((3, 16)), rng.standard_normal((11, 16)), rng.standard_normal((11, 16))
    o, lse = O.attention(q, K, V)
    for h in range(3):
        s = [sum(q[h, i] * K[t, i] for i in range(16)) / 4.0 for t in range(11)]
        L = math.log(sum(math.exp(v) for v in s))
        assert abs(L - lse[h]) < 1e-12
        for j in range(16):
            want = sum(math.exp(s[t] - L) * V[t, j] for t in range(11))
            assert abs(want - o[h, j]) < 1e-12


def test_attention_special_cases():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((2, 128))
    K = np.tile(rng.standard_normal(128), (7, 1))
    V = rng.standard_normal((7, 128))
    o, _ = O.attention(q, K, V)
    np.testing.assert_allclose(o, np.tile(V.mean(0), (2, 1)), rtol=1e-12, atol=1e-12)
    o1, lse1 = O.attention(q, K[:1], V[:1])
    np.testing.assert_allclose(o1, np.tile(V[0], (2, 1)), rtol=1e-14)
    np.testing.assert_allclose(lse1, q @ K[0] / math.sqrt(128), rtol=1e-12)


# ---------------------------------------------------------------- zones
def test_zone_bounds():
    assert O.zone_bounds(1) == (1, 64)
    assert O.zone_bounds(64) == (64, 64)
    assert O.zone_bounds(320) == (64, 64)
    assert O.zone_bounds(321) == (64, 65)
    s, F = O.zone_bounds(2048)
    assert F - 64 == 1728 and 2048 - F == 256  # 64 sink + 1728 INT2 + 256 recent
    assert O.zone_bounds(32800, shared=32768) == (64, 32768)
    assert O.zone_bounds(40000, shared=32768) == (64, 40000 - 256)


# ---------------------------------------------------------------- P8: storage vs the pages
def test_storage_numbers_match_pages():
    g = json.load(open(GOLDEN))
    assert O.SINK == g["sink_tokens"]["value"] and O.RECENT == g["recent_tokens"]["value"]
    assert O.pack_codes(np.zeros(128, np.uint8)).size * g["codes_per_byte"]["value"] == 128
    assert round(100 * (O.SINK + O.RECENT) / 131072, 2) == g["bf16_share_of_128k_percent"]["value"]
    assert O.history_bits_per_element(128) == 2.25 == g["bpe_int2_history_baselines"]["value"]
    assert round(O.bits_per_element(g["bpe_long_context_128k"]["context"]), 2) == g["bpe_long_context_128k"]["value"]
    assert round(O.bits_per_element(g["bpe_32k"]["context"]), 2) == g["bpe_32k"]["value"]
    # group 32 would not give the printed numbers
    assert round(O.bits_per_element(131072, group_size=32), 2) != g["bpe_long_context_128k"]["value"]
    assert 16 / 2 == g["kv_memory_reduction_vs_bf16_history"]["value"]
    assert 7.0 < 16 / O.history_bits_per_element(128) < 8.0


# ---------------------------------------------------------------- P9: decode end to end
def _grid_rows(rng, n, G):
    s = np.float32(2.0 ** rng.integers(-3, 1))
    z = np.float32(-1.5)
    k = rng.integers(0, 4, size=(n, 128))
    k[:, ::G] = 0
    k[:, 1::G] = 3
    return k.astype(np.uint8), np.full((n, 128 // G), s, np.float16), np.full((n, 128 // G), z, np.float16)


@pytest.mark.parametrize("G,absorbed", [(128, False), (32, False), (128, True)])
def test_decode_reference_equals_attention_in_original_basis(basis, G, absorbed):
    """INT2 tokens with dequantised rotated rows r are the original-basis rows r R^T:
    decode_reference must equal plain attention over those rows."""
    rng = np.random.default_rng(10)
    U_k = basis[0]
    U_v = W.synthetic_basis(0, 0, 0, 1)[0]
    R_k, R_v = O.rotation_matrix(U_k), O.rotation_matrix(U_v)
    q = rng.standard_normal((4, 128))
    kb, vb = rng.standard_normal((30, 128)), rng.standard_normal((30, 128))
    ck, sk, zk = _grid_rows(rng, 50, G)
    cv, sv, zv = _grid_rows(rng, 50, G)
    o, lse = O.decode_reference(q, kb, vb, ck, sk, zk, cv, sv, zv, U_k, U_v, G, absorbed)
    k_orig = O.dequantize(ck, sk, zk, G) @ R_k.T
    v_deq = O.dequantize(cv, sv, zv, G)
    v_orig = v_deq if absorbed else v_deq @ R_v.T
    # R_k is orthogonal to ~1e-7 (fp32 U), so q.(r R^T) and (qR).r agree to ~1e-6
    o_ref, lse_ref = O.attention(q, np.vstack([kb, k_orig]), np.vstack([vb, v_orig]))
    np.testing.assert_allclose(o, o_ref, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5)


def test_decode_reference_identity_rotation_equals_bf16_path():
    """R = I (U = P H), clip 1, grid-exact rows: the INT2 path reproduces the BF16 path exactly."""
    rng = np.random.default_rng(11)
    U_id = O.bitrev_matrix() @ O.hadamard()  # U H P = P H H P = I
    np.testing.assert_allclose(O.rotation_matrix(U_id), np.eye(128), atol=1e-14)
    q = rng.standard_normal((4, 128))
    ck, sk, zk = _grid_rows(rng, 40, 128)
    cv, sv, zv = _grid_rows(rng, 40, 128)
    k = O.dequantize(ck, sk, zk, 128)
    v = O.dequantize(cv, sv, zv, 128)
    enc = O.encode_rows(k, U_id, 1.0, 128)
    np.testing.assert_array_equal(enc["codes"], ck)
    o_int2, _ = O.decode_reference(q, k[:0], v[:0], ck, sk, zk, cv, sv, zv, U_id, U_id, 128)
    o_bf16, _ = O.decode_reference(q, k, v, ck[:0], sk[:0], zk[:0], cv[:0], sv[:0], zv[:0], U_id, U_id, 128)
    np.testing.assert_allclose(o_int2, o_bf16, rtol=1e-12, atol=1e-12)


def test_encode_rows_rotation_then_quantise(basis):
    rng = np.random.default_rng(12)
    x = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((8, 128)).astype(np.float32)))
    enc = O.encode_rows(x, basis[0], 0.9, 128)
    np.testing.assert_allclose(enc["rot64"], x.astype(np.float64) @ O.rotation_matrix(basis[0]), rtol=1e-12)
    c2, s2, z2, _ = O.quantize_fp32(enc["rot64"].astype(np.float32), np.float32(0.9), 128)
    np.testing.assert_array_equal(enc["codes"], c2)


# ---------------------------------------------------------------- Lloyd-Max codebook variant
# (symmetric levels (0, a, 3 - a, 3) in the uniform quantiser's group frame; a = 1 is uniform)

def test_lloyd_at_a1_is_the_uniform_quantiser_including_ties():
    rng = np.random.default_rng(11)
    r = (rng.standard_normal((300, 128)) * np.where(rng.random(128) < 0.05, 20, 1)).astype(np.float32)
    for clip in (np.float32(0.9), np.float32(1.0)):
        a = O.quantize_fp32(r, clip, 32)
        b = O.quantize_lloyd_fp32(r, clip, 32, 1.0)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)
    # exact ties at u = 0.5, 1.5, 2.5 (group min 0, max 3, c = 1: s = 1, z = 0)
    g = np.zeros(128, np.float32)
    g[1], g[2:5] = 3.0, (0.5, 1.5, 2.5)
    codes, s16, z16, _ = O.quantize_lloyd_fp32(g[None], np.float32(1.0), 128, 1.0)
    assert float(s16[0, 0]) == 1.0 and float(z16[0, 0]) == 0.0
    assert codes[0, 2:5].tolist() == [0, 2, 2]  # ties to even, as rint
    np.testing.assert_array_equal(O.dequantize_lloyd(codes, s16, z16, 128, 1.0), O.dequantize(codes, s16, z16, 128))


def test_lloyd_codes_are_the_nearest_level():
    rng = np.random.default_rng(12)
    r = rng.standard_normal((400, 128)).astype(np.float32)
    for a in (0.7, 1.0, 1.23):
        codes, s16, z16, _ = O.quantize_lloyd_fp32(r, np.float32(0.9), 128, a)
        u = O.normalized_rows(r, np.float32(0.9), 128).astype(np.float64)
        lv = O.lloyd_levels(a).astype(np.float64)
        dist = np.abs(u[..., None] - lv)
        best = dist.argmin(axis=-1)
        tie = np.sort(dist, axis=-1)[..., 1] - np.sort(dist, axis=-1)[..., 0] < 1e-6
        assert np.all((codes == best) | tie)


def test_lloyd_fit_uniform_density_gives_equal_spacing():
    u = np.random.default_rng(13).uniform(0.0, 3.0, 2_000_000)
    assert abs(O.lloyd_fit(u) - 1.0) < 3e-3


def test_lloyd_fit_triangular_density_closed_form():
    """Density on [0, 3] proportional to 1.5 - |u - 1.5|. The centroid of the cell (a/2, 1.5) of
    level a under density u is (2/3) (1.5^3 - x^3) / (1.5^2 - x^2) with x = a/2; the fixed point,
    found by a root finder, is the codebook Lloyd's algorithm must reach (the mirrored cell gives
    the same equation by symmetry)."""
    from scipy.optimize import brentq
    f = lambda a: (2.0 / 3.0) * (1.5 ** 3 - (a / 2) ** 3) / (1.5 ** 2 - (a / 2) ** 2) - a  # noqa: E731
    a_star = brentq(f, 0.1, 1.45)
    rng = np.random.default_rng(14)
    u = rng.triangular(0.0, 1.5, 3.0, 4_000_000)
    assert abs(O.lloyd_fit(u, iters=200) - a_star) < 3e-3
    assert a_star > 1.0  # mass concentrated in the middle pulls the interior levels inward


def test_lloyd_fit_lowers_the_reconstruction_error():
    rng = np.random.default_rng(15)
    r = rng.standard_normal((2000, 128)).astype(np.float32)
    a = O.lloyd_fit(O.normalized_rows(r, np.float32(0.9), 128))
    err = {}
    for aa in (1.0, a):
        c, s, z, _ = O.quantize_lloyd_fp32(r, np.float32(0.9), 128, aa)
        err[aa] = np.mean((O.dequantize_lloyd(c, s, z, 128, aa) - r) ** 2)
    assert a != 1.0 and err[a] < err[1.0]


# ---------------------------------------------------------------- Lloyd-Max branch of the decode
def _literal_level(code, a):
    """Level of a 2-bit code in the Lloyd-Max codebook, typed out as the table (0, a, 3 - a, 3);
    3 - a is formed in fp32, the precision the codebook's levels are specified in."""
    a = np.float32(a)
    return {0: 0.0, 1: float(a), 2: float(np.float32(3.0) - a), 3: 3.0}[int(code)]


def test_decode_reference_lloyd_codebook_against_brute_force_rows(basis):
    """decode_reference(codebook=(a_K, a_V)) equals plain attention over INT2 rows rebuilt
    element by element from the literal level table and brought back by R^T; a_K != a_V, so the
    K and V levels swapped, or the uniform levels, give a different result."""
    rng = np.random.default_rng(21)
    G = 32
    U_k = basis[0]
    U_v = W.synthetic_basis(0, 0, 0, 1)[0]
    R_k, R_v = O.rotation_matrix(U_k), O.rotation_matrix(U_v)
    a_k, a_v = np.float32(0.62), np.float32(1.31)
    n = 24
    ck = rng.integers(0, 4, size=(n, 128)).astype(np.uint8)
    cv = rng.integers(0, 4, size=(n, 128)).astype(np.uint8)
    sk = (rng.uniform(0.2, 1.5, size=(n, 128 // G))).astype(np.float16)
    sv = (rng.uniform(0.2, 1.5, size=(n, 128 // G))).astype(np.float16)
    zk = (rng.uniform(-2.0, -0.5, size=(n, 128 // G))).astype(np.float16)
    zv = (rng.uniform(-2.0, -0.5, size=(n, 128 // G))).astype(np.float16)
    k_rot = np.zeros((n, 128))
    v_rot = np.zeros((n, 128))
    for t in range(n):
        for j in range(128):
            g = j // G
            k_rot[t, j] = float(zk[t, g]) + float(sk[t, g]) * _literal_level(ck[t, j], a_k)
            v_rot[t, j] = float(zv[t, g]) + float(sv[t, g]) * _literal_level(cv[t, j], a_v)
    q = rng.standard_normal((4, 128))
    kb, vb = rng.standard_normal((5, 128)), rng.standard_normal((5, 128))
    o_ref, lse_ref = O.attention(q, np.vstack([kb, k_rot @ R_k.T]), np.vstack([vb, v_rot @ R_v.T]))
    o, lse = O.decode_reference(q, kb, vb, ck, sk, zk, cv, sv, zv, U_k, U_v, G, codebook=(a_k, a_v))
    np.testing.assert_allclose(o, o_ref, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5)
    for wrong in ((a_v, a_k), (np.float32(1.0), np.float32(1.0))):
        o_w, _ = O.decode_reference(q, kb, vb, ck, sk, zk, cv, sv, zv, U_k, U_v, G, codebook=wrong)
        assert np.abs(o_w - o_ref).max() > 1e-2


def test_dequantize_lloyd_matches_literal_table():
    """Every code of every group against the literal table, for a few a (including a = 1, where the
    table is the uniform levels 0, 1, 2, 3)."""
    codes = np.tile(np.arange(4, dtype=np.uint8), 32)[None]
    s16 = np.array([[0.5, 0.25, 2.0, 1.0]], np.float16)
    z16 = np.array([[-1.0, 0.5, -3.0, 0.0]], np.float16)
    for a in (0.55, 1.0, 1.4):
        got = O.dequantize_lloyd(codes, s16, z16, 32, a)
        for j in range(128):
            g = j // 32
            want = float(z16[0, g]) + float(s16[0, g]) * _literal_level(codes[0, j], np.float32(a))
            assert got[0, j] == want
    np.testing.assert_array_equal(O.dequantize_lloyd(codes, s16, z16, 32, 1.0), O.dequantize(codes, s16, z16, 32))


# ---------------------------------------------------------------- zones with a shared prefix
def _simulate_zones(events, sink=64, recent=256):
    """Token-level model of one sequence's cache, written from the serving description without the
    frontier formula: positions below `sink` stay BF16; a sharer starts with positions
    [sink, shared) already INT2 (the owner's pages) and an empty recent window; every appended
    token enters a FIFO recent window of `recent` slots and pushes the oldest one into INT2 history
    when the window overflows. events: ("start", shared) then ("append", n) items. Returns the
    first recent position after each append (the position the INT2 history ends at)."""
    L, fifo, out = 0, [], []
    for kind, n in events:
        if kind == "start":
            L = n
            fifo = []
            continue
        for _ in range(n):
            pos = L
            L += 1
            if pos < sink:
                continue
            fifo.append(pos)
            if len(fifo) > recent:
                fifo.pop(0)
        out.append((L, fifo[0] if fifo else max(sink, L) if L <= sink else L))
    return out


@pytest.mark.parametrize("shared", [0, 64, 64 + 64 * 7, 32768])
def test_zone_bounds_shared_prefix_against_token_model(shared):
    """zone_bounds(L, shared) against the token-level model above, for a fresh sequence (shared = 0)
    and for sharers of a prefix of `shared` tokens, over appends that cross the recent window's size
    and page boundaries; the history of a sharer always covers the owner's shared pages."""
    start = [("start", shared)] if shared else []
    steps = [1, 1, 62, 1, 190, 1, 1, 3, 64, 64, 1, 200, 127, 1, 1]
    model = _simulate_zones(start + [("append", n) for n in steps])
    for L, first_recent in model:
        sink_end, F = O.zone_bounds(L, shared=shared)
        assert sink_end == min(64, L)
        assert F == max(64, first_recent) if L > 64 else F == 64
        if shared:
            assert F >= shared  # the shared pages [64, shared) stay INT2 history
            n_shared_pages = (shared - 64) // 64
            assert (F - 64 + 63) // 64 >= n_shared_pages
