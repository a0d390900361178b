"""OSCAR INT2 paged-KV decode: CPU oracle (numpy; fp64 except the fp32 quantiser).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources (page title, then section / paragraph):
  [snilld]  "OSCAR fra Together AI goer 2-bit KV-cache mere praktisk" (snilld.dk)
  [arddev]  "oscar-2bit-kv-cache" news summary (arddev.tech)
  [author]  OSCAR author write-up by Zhongzhu Zhou (m.th-motor.com), one long
            paragraph sequence; cited by its topic and the figure it describes.

What the method computes, as restated here:
  * Keys and values are rotated before INT2 quantisation by R = U . H . P, per
    layer and per KV head: U aligns with the attention statistics, H is the
    Walsh-Hadamard transform, P a bit-reversal permutation ([author] rotation
    paragraph; [arddev] "Аналитика" lists the order: covariance alignment, then
    Walsh-Hadamard, then bit-reversal; [snilld] "Hvad OSCAR gør anderledes").
  * Rotated rows are clipped and quantised to 2 bits with a per-group scale and
    zero point, four codes per byte ([author] serving paragraph and the
    rotation paragraph on clipping thresholds).
  * Decode attends over BF16 sink/recent tokens and INT2 history; the two
    results are combined by an online-softmax merge ([author] serving
    paragraph). Keys are compared in the rotated basis, which preserves dot
    products because R is orthogonal.

Readings where the pages are silent (each is listed in the design notes):
row-vector convention x_rot = x . R; Sylvester-ordered, orthonormal H of size
128; a single 7-bit bit-reversal over head_dim; groups run along head_dim after
rotation; clip ratio c scales the group min and max; zero point = clipped min,
x_hat = code * s + z with fp16 s and z; codes computed from the fp16-rounded
s, z with IEEE fp32 subtraction and division and round-half-even; little-endian
2-bit packing; softmax scale 1/sqrt(head_dim).
"""
from __future__ import annotations

import math
import struct

import numpy as np

__all__ = [
    "HEAD_DIM", "SINK", "RECENT", "PAGE",
    "hadamard", "bitrev", "bitrev_matrix", "rotation_matrix", "rotate_rows",
    "half_rn", "quantize_fp32", "pack_codes", "unpack_codes", "dequantize",
    "lloyd_levels", "normalized_rows", "quantize_lloyd_fp32", "dequantize_lloyd", "lloyd_fit",
    "attention", "merge_segments", "zone_bounds", "encode_rows", "decode_reference",
    "history_bits_per_element", "bits_per_element", "fp16_bits_python",
]

HEAD_DIM = 128
SINK = 64      # [snilld] "Hvad vi ved om resultaterne"; [arddev] "Аналитика" (first 64 tokens BF16)
RECENT = 256   # [arddev] "Аналитика" (last 256 tokens BF16); "Как применить сегодня" (CLI flags)
PAGE = 64      # page size of the synthetic workloads


# --------------------------------------------------------------------------------------------
# Transforms: H, P, R = U H P  ([author] rotation paragraph; [arddev] "Аналитика")
# --------------------------------------------------------------------------------------------

def hadamard(d: int = HEAD_DIM) -> np.ndarray:
    """Orthonormal Walsh-Hadamard matrix in natural (Sylvester) order:
    H[i, j] = (-1)^popcount(i & j) / sqrt(d)."""
    i = np.arange(d).reshape(-1, 1)
    j = np.arange(d).reshape(1, -1)
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    return np.where(pc % 2 == 0, 1.0, -1.0) / math.sqrt(d)


def bitrev(i: int, nbits: int) -> int:
    """Reverse the low ``nbits`` bits of ``i``."""
    r = 0
    for b in range(nbits):
        if i >> b & 1:
            r |= 1 << (nbits - 1 - b)
    return r


def bitrev_matrix(d: int = HEAD_DIM) -> np.ndarray:
    """Permutation P with (y P)_j = y_{bitrev(j)}, i.e. P[i, j] = [i == bitrev(j)]."""
    nbits = int(round(math.log2(d)))
    P = np.zeros((d, d))
    for j in range(d):
        P[bitrev(j, nbits), j] = 1.0
    return P


def rotation_matrix(U) -> np.ndarray:
    """Composite rotation R = U . H . P in fp64 from the fp32 basis U (rows act on x: x_rot = x R)."""
    U = np.asarray(U, dtype=np.float64)
    d = U.shape[0]
    return U @ hadamard(d) @ bitrev_matrix(d)


def rotate_rows(x, R) -> np.ndarray:
    """x_rot = x . R for row vectors, fp64."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(R, dtype=np.float64)


# --------------------------------------------------------------------------------------------
# Quantiser (fp32 spec, every step one IEEE round-to-nearest-even operation)
# ([author] serving paragraph: clip, asymmetric scale/zero point, 4 codes per byte)
# --------------------------------------------------------------------------------------------

def half_rn(x) -> np.ndarray:
    """fp32 -> fp16, round to nearest even (numpy's conversion; overflow gives inf)."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float32).astype(np.float16)


def quantize_fp32(r, clip, group_size: int):
    """Quantise fp32 rotated rows to 2-bit codes, per group along head_dim.

    For every group: mn, mx = group min and max; lo = c*mn; hi = c*mx;
    s = (hi - lo) / 3; s16 = fp16(s); z16 = fp16(lo); with sf, zf their fp32
    values: code = clamp(rint((x - zf) / sf), 0, 3), or 0 for the whole group
    when sf == 0. All arithmetic is fp32. A group whose s or lo is non-finite or
    overflows fp16 is flagged in ``bad``.

    r: float32 [..., d]; clip: fp32 scalar (or broadcastable to [...]).
    Returns codes uint8 [..., d], s16 float16 [..., d/G], z16 float16 [..., d/G], bad bool [..., d/G].
    """
    r = np.asarray(r, dtype=np.float32)
    d = r.shape[-1]
    assert d % group_size == 0
    g = r.reshape(*r.shape[:-1], d // group_size, group_size)
    c = np.asarray(clip, dtype=np.float32)
    if c.ndim:
        c = c[..., None]
    mn = g.min(axis=-1)
    mx = g.max(axis=-1)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        lo = (c * mn).astype(np.float32)
        hi = (c * mx).astype(np.float32)
        s32 = ((hi - lo) / np.float32(3.0)).astype(np.float32)
        s16 = half_rn(s32)
        z16 = half_rn(lo)
        sf = s16.astype(np.float32)
        zf = z16.astype(np.float32)
        bad = ~np.isfinite(s32) | ~np.isfinite(lo) | ~np.isfinite(sf) | ~np.isfinite(zf)
        t = ((g - zf[..., None]).astype(np.float32) / sf[..., None]).astype(np.float32)
        code = np.clip(np.rint(t), 0.0, 3.0)
    code = np.where((sf == 0)[..., None] | ~np.isfinite(code), 0.0, code)
    return code.astype(np.uint8).reshape(r.shape), s16, z16, bad


def pack_codes(codes) -> np.ndarray:
    """Canonical packing: byte j>>2 holds code j in bits 2*(j&3) .. 2*(j&3)+1 (4 codes per byte)."""
    c = np.asarray(codes, dtype=np.uint8)
    d = c.shape[-1]
    q = c.reshape(*c.shape[:-1], d // 4, 4).astype(np.uint32)
    b = q[..., 0] | (q[..., 1] << 2) | (q[..., 2] << 4) | (q[..., 3] << 6)
    return b.astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    """Inverse of :func:`pack_codes`."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.stack([(p >> (2 * k)) & 3 for k in range(4)], axis=-1)
    return out.reshape(*p.shape[:-1], p.shape[-1] * 4).astype(np.uint8)


def dequantize(codes, s16, z16, group_size: int) -> np.ndarray:
    """x_hat = code * s + z (exact in fp64), s, z per group."""
    codes = np.asarray(codes, dtype=np.float64)
    d = codes.shape[-1]
    s = np.repeat(np.asarray(s16, dtype=np.float64), group_size, axis=-1)
    z = np.repeat(np.asarray(z16, dtype=np.float64), group_size, axis=-1)
    assert s.shape[-1] == d
    return codes * s + z


# --------------------------------------------------------------------------------------------
# Lloyd-Max codebook variant ([author] closing paragraph: the newest codebase brings a Lloyd-Max
# codebook into the attention-aware rotation). Reading: the group frame of the uniform quantiser
# is kept (same lo, hi, fp16 s and z, same storage); the four levels become (0, a, 3 - a, 3)
# instead of (0, 1, 2, 3), with one a per (layer, KV head, K|V) fitted by Lloyd's algorithm
# (nearest-level cells, then centroids) with the end levels held at the clipped min and max and
# the codebook kept symmetric. a = 1 is the uniform quantiser.
# --------------------------------------------------------------------------------------------

def lloyd_levels(a) -> np.ndarray:
    """The four levels (0, a, 3 - a, 3) of the symmetric codebook, in fp32."""
    a = np.float32(a)
    return np.array([0.0, a, np.float32(3.0) - a, 3.0], dtype=np.float32)


def normalized_rows(r, clip, group_size: int):
    """u = (x - zf) / sf of fp32 rotated rows in their group's frame (fp32, as in quantize_fp32);
    groups with sf == 0 give 0. Returns u float32 [..., d]."""
    r = np.asarray(r, dtype=np.float32)
    d = r.shape[-1]
    g = r.reshape(*r.shape[:-1], d // group_size, group_size)
    c = np.float32(clip)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        lo = (c * g.min(axis=-1)).astype(np.float32)
        hi = (c * g.max(axis=-1)).astype(np.float32)
        s16 = half_rn(((hi - lo) / np.float32(3.0)).astype(np.float32))
        zf = half_rn(lo).astype(np.float32)
        sf = s16.astype(np.float32)
        u = ((g - zf[..., None]).astype(np.float32) / sf[..., None]).astype(np.float32)
    u = np.where((sf == 0)[..., None] | ~np.isfinite(u), np.float32(0), u)
    return u.reshape(r.shape)


def quantize_lloyd_fp32(r, clip, group_size: int, a):
    """Lloyd-Max variant of quantize_fp32: same lo, hi, s16, z16 and u = (x - zf) / sf (fp32);
    the code is the nearest level of (0, a, 3 - a, 3):
        code = [u > t0] + [u >= t1] + [u > t2],  t0 = a * 0.5, t1 = 1.5, t2 = 3 - a * 0.5 (fp32),
    which at a = 1 is clamp(rint(u), 0, 3) with ties to even. Returns (codes, s16, z16, bad)."""
    codes_u, s16, z16, bad = quantize_fp32(r, clip, group_size)
    u = normalized_rows(r, clip, group_size)
    a = np.float32(a)
    t0 = (a * np.float32(0.5)).astype(np.float32)
    t1 = np.float32(1.5)
    t2 = (np.float32(3.0) - t0).astype(np.float32)
    code = (u > t0).astype(np.uint8) + (u >= t1).astype(np.uint8) + (u > t2).astype(np.uint8)
    sf = np.repeat(s16.astype(np.float32), group_size, axis=-1).reshape(code.shape)
    code = np.where(sf == 0, np.uint8(0), code)
    return code.astype(np.uint8), s16, z16, bad


def dequantize_lloyd(codes, s16, z16, group_size: int, a) -> np.ndarray:
    """x_hat = z + s * level[code] (fp64) with level = (0, a, 3 - a, 3) from fp32 a."""
    lv = lloyd_levels(a).astype(np.float64)
    codes = np.asarray(codes, dtype=np.int64)
    s = np.repeat(np.asarray(s16, dtype=np.float64), group_size, axis=-1)
    z = np.repeat(np.asarray(z16, dtype=np.float64), group_size, axis=-1)
    return lv[codes] * s + z


def lloyd_fit(u, iters: int = 50, a0: float = 1.0, tol: float = 1e-9) -> float:
    """Lloyd's algorithm for the interior level a of the codebook (0, a, 3 - a, 3) on samples u of
    the group frame (fp64): assign every sample to its nearest level, then move a to the centroid
    of the samples of level a together with the mirror images 3 - u of the samples of level 3 - a
    (the codebook stays symmetric; the end levels stay fixed). a is kept in [0.05, 1.45]."""
    u = np.asarray(u, dtype=np.float64).ravel()
    a = float(a0)
    for _ in range(iters):
        t0, t2 = a / 2.0, 3.0 - a / 2.0
        c1 = u[(u > t0) & (u < 1.5)]
        c2 = u[(u >= 1.5) & (u <= t2)]
        n = c1.size + c2.size
        if n == 0:
            break
        new = (c1.sum() + (3.0 - c2).sum()) / n
        new = min(1.45, max(0.05, new))
        if abs(new - a) < tol:
            a = new
            break
        a = new
    return a


# --------------------------------------------------------------------------------------------
# Attention and the online-softmax merge ([author] serving paragraph)
# --------------------------------------------------------------------------------------------

def attention(q, K, V, scale=None):
    """Softmax attention of query rows q [h, d] over keys K [n, d] / values V [n, d], fp64.

    One pass over all n tokens with max subtraction. Returns (o [h, d], lse [h])
    with lse the natural-log sum of exp(score). n == 0 gives o = 0, lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[-1] if V.ndim == 2 else d)), np.full(q.shape[0], -np.inf)
    s = (q @ K.T) * scale
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e @ V) / l
    return o, (m + np.log(l))[:, 0]


def merge_segments(parts):
    """Combine per-segment results (o_i normalised, lse_i) into the softmax over the union:
    M = max lse_i, w_i = exp(lse_i - M), o = sum w_i o_i / sum w_i, lse = M + log sum w_i.
    Segments with lse = -inf contribute nothing."""
    lses = np.stack([p[1] for p in parts], axis=0)
    M = lses.max(axis=0)
    Ms = np.where(np.isfinite(M), M, 0.0)
    w = np.exp(lses - Ms)
    den = w.sum(axis=0)
    num = sum(w[i][:, None] * parts[i][0] for i in range(len(parts)))
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(den[:, None] > 0, num / np.where(den > 0, den, 1.0)[:, None], 0.0)
        lse = np.where(den > 0, Ms + np.log(np.where(den > 0, den, 1.0)), -np.inf)
    return o, lse


# --------------------------------------------------------------------------------------------
# Cache-state model ([author] serving paragraph: new token to recent, oldest recent demoted;
# sink and recent BF16, rest INT2; [arddev] "Аналитика": 64 + 256 BF16 tokens)
# --------------------------------------------------------------------------------------------

def zone_bounds(L: int, shared: int = 0, sink: int = SINK, recent: int = RECENT):
    """Zones of a sequence holding positions [0, L):
    sink = [0, min(sink, L)); INT2 = [sink, F); recent = [F, L), with the demote
    frontier F = max(sink, shared, L - recent). ``shared`` is the length of a
    prefix whose INT2 pages are shared with another sequence (0 if none).
    Returns (sink_end, F)."""
    F = max(sink, shared, L - recent)
    return min(sink, L), F


# --------------------------------------------------------------------------------------------
# Encode (demote) and decode for one (sequence, layer, KV head)
# --------------------------------------------------------------------------------------------

def encode_rows(x, U, clip, group_size: int, rotate: bool = True):
    """Demote rows x (bf16 values as float) : rotate by R in fp64, round the rows to fp32,
    quantise with the fp32 spec. Returns dict(rot64, rot32, codes, s16, z16, bad)."""
    x = np.asarray(x, dtype=np.float64)
    rot64 = rotate_rows(x, rotation_matrix(U)) if rotate else x.copy()
    rot32 = rot64.astype(np.float32)
    codes, s16, z16, bad = quantize_fp32(rot32, np.float32(clip), group_size)
    return dict(rot64=rot64, rot32=rot32, codes=codes, s16=s16, z16=z16, bad=bad)


def decode_reference(q, k_bf16, v_bf16, codes_k, s_k, z_k, codes_v, s_v, z_v,
                     U_k, U_v, group_size: int, v_rot_absorbed: bool = False, codebook=None):
    """Decode attention for the query heads of one KV head, over the union of
    BF16 tokens (sink + recent: k_bf16, v_bf16 [n_b, d]) and INT2 tokens
    (codes [n_i, d], fp16 s, z [n_i, d/G]).

    Keys: BF16 scores use raw q; INT2 scores use q_rot = q R_K against the
    dequantised rotated keys. Values: INT2 values are dequantised and brought
    back to the original basis by R_V^T (skipped when the value rotation is
    absorbed into the projection weights, [arddev] "Аналитика"). One-pass
    softmax over all tokens with scale 1/sqrt(d), fp64.
    codebook = (a_K, a_V) dequantises INT2 codes with the Lloyd-Max levels (0, a, 3 - a, 3)
    instead of (0, 1, 2, 3).
    Returns (o [h, d], lse [h]).
    """
    q = np.asarray(q, dtype=np.float64)
    R_k = rotation_matrix(U_k)
    R_v = rotation_matrix(U_v)
    q_rot = q @ R_k
    if codebook is None:
        k_hat = dequantize(codes_k, s_k, z_k, group_size)
        v_hat = dequantize(codes_v, s_v, z_v, group_size)
    else:
        k_hat = dequantize_lloyd(codes_k, s_k, z_k, group_size, codebook[0])
        v_hat = dequantize_lloyd(codes_v, s_v, z_v, group_size, codebook[1])
    if not v_rot_absorbed:
        v_hat = v_hat @ R_v.T
    d = q.shape[-1]
    scale = 1.0 / math.sqrt(d)
    s_b = (q @ np.asarray(k_bf16, dtype=np.float64).T) * scale
    s_i = (q_rot @ k_hat.T) * scale
    s = np.concatenate([s_b, s_i], axis=1)
    V = np.concatenate([np.asarray(v_bf16, dtype=np.float64), v_hat], axis=0)
    if s.shape[1] == 0:
        return np.zeros((q.shape[0], d)), np.full(q.shape[0], -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return (e @ V) / l, (m + np.log(l))[:, 0]


# --------------------------------------------------------------------------------------------
# Storage accounting ([arddev] "Аналитика": 2.28 bits per element, 0.24% BF16 at 128K;
# [author] Fig. 3 / Fig. 4 paragraphs: 2.28 and 2.38 BPE)
# --------------------------------------------------------------------------------------------

def history_bits_per_element(group_size: int, d: int = HEAD_DIM, scale_bits: int = 16) -> float:
    """INT2 history storage: 2 bits per element plus an fp16 scale and fp16 zero per group."""
    return (2 * d + 2 * scale_bits * (d // group_size)) / d


def bits_per_element(L: int, group_size: int = 128, d: int = HEAD_DIM,
                     sink: int = SINK, recent: int = RECENT) -> float:
    """Average stored bits per KV element of a length-L context: BF16 (16 bits) for
    the sink and recent tokens, INT2 history for the rest."""
    n_bf16 = min(L, sink + recent)
    n_int2 = L - n_bf16
    return (16.0 * n_bf16 + history_bits_per_element(group_size, d) * n_int2) / L


def fp16_bits_python(x: float) -> int:
    """fp16 bit pattern of a Python float via the struct module (IEEE round-half-even);
    an independent route used to pin :func:`half_rn`."""
    return struct.unpack("<H", struct.pack("<e", x))[0]
