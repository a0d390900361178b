"""Counter-based synthetic inputs (host side).

Every K/V/q element is a pure function of (seed, tag, seq, layer, head, kv,
pos, dim), so any slice of a workload can be regenerated on the host after the
device generator (``synth.cu``, same definition) has filled a cache with it.

Generator definition
--------------------
* Hash: the SplitMix64 output function of Steele, Lea and Flood, "Fast
  splittable pseudorandom number generators" (OOPSLA 2014), used as a
  counter-based generator: ``h(n) = mix64(seed + (n + 1) * 0x9E3779B97F4A7C15)``
  (all arithmetic mod 2**64), with ``mix64(z)``: ``z ^= z >> 30; z *=
  0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31``.
* Counter ``n`` packs the element coordinates into bit fields
  (tag:4 | seq:10 | layer:7 | head:6 | kv:1 | pos:20 | dim:7, low bits last).
* Normal draw: Irwin-Hall sum of the four 16-bit fields of ``h``
  (``S = u0+u1+u2+u3``), centred and scaled in fp32:
  ``z = float32(S - 131070) * float32(1/sigma)``, ``sigma**2 = (65536**2-1)/3``.
  All steps are integer-exact except one fp32 multiply (IEEE round to nearest
  even), so host and device agree bit for bit. Outlier channels use the scale
  ``float32(20/sigma)`` instead (one rounding of the fp64 product).
* bf16: round-to-nearest-even of the fp32 value.

The distribution is a 4-term Irwin-Hall approximation of N(0, 1) (bounded at
+-3.46 sigma); it stands in for the pages' "N(0,1) with channel outliers".
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "GOLDEN", "mix64", "counter_index", "hash64", "INV_SIGMA_F32", "OUTLIER_SCALE_F32",
    "TAG_KV", "TAG_Q", "TAG_OUTLIER",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "normal_f32_from_hash",
    "kv_rows_bf16", "q_rows_bf16", "outlier_mask_bernoulli", "outlier_mask_exact",
    "synthetic_basis", "aligned_query_rows", "config4_lengths", "Config", "CONFIGS",
]

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TAG_KV = 0
TAG_Q = 1
TAG_OUTLIER = 2

_SIGMA = math.sqrt((65536.0 ** 2 - 1.0) / 3.0)
INV_SIGMA_F32 = np.float32(1.0 / _SIGMA)
OUTLIER_SCALE_F32 = np.float32(20.0 / _SIGMA)
IH_CENTER = 131070  # 4 * 65535 / 2


def mix64(z):
    """SplitMix64 output mixing of a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z ^ (z >> np.uint64(30))
        z = z * _M1
        z = z ^ (z >> np.uint64(27))
        z = z * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def counter_index(tag, seq, layer, head, kv, pos, dim):
    """Pack element coordinates into the 55-bit counter (see module doc)."""
    u = lambda v: np.asarray(v, dtype=np.uint64)  # noqa: E731
    return ((u(tag) << np.uint64(51)) | (u(seq) << np.uint64(41)) | (u(layer) << np.uint64(34))
            | (u(head) << np.uint64(28)) | (u(kv) << np.uint64(27)) | (u(pos) << np.uint64(7))
            | u(dim))


def hash64(seed, n):
    """Counter-based SplitMix64: the (n+1)-th output of a stream seeded with ``seed``."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (np.asarray(n, dtype=np.uint64) + np.uint64(1)) * GOLDEN
    return mix64(z)


def normal_f32_from_hash(h, scale_f32):
    """Irwin-Hall(4) draw from a uint64 hash, times an fp32 scale (one rounding)."""
    h = np.asarray(h, dtype=np.uint64)
    m = np.uint64(0xFFFF)
    s = ((h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m)
         + ((h >> np.uint64(48)) & m)).astype(np.int64) - IH_CENTER
    return s.astype(np.float32) * np.float32(scale_f32)


def f32_to_bf16_bits(x):
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((b + r) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def kv_rows_bf16(seed, seq_key, layer, head, kv, positions, outlier_mask, head_dim=128):
    """bf16 bit patterns of K (kv=0) or V (kv=1) rows, shape [len(positions), head_dim].

    ``outlier_mask``: bool [head_dim] for this (layer, head, kv); outlier channels
    are drawn with the x20 scale.
    """
    pos = np.asarray(positions, dtype=np.uint64).reshape(-1, 1)
    dim = np.arange(head_dim, dtype=np.uint64).reshape(1, -1)
    n = counter_index(TAG_KV, seq_key, layer, head, kv, pos, dim)
    h = hash64(seed, n)
    scale = np.where(np.asarray(outlier_mask, dtype=bool).reshape(1, -1),
                     OUTLIER_SCALE_F32, INV_SIGMA_F32).astype(np.float32)
    m = np.uint64(0xFFFF)
    s = ((h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m)
         + ((h >> np.uint64(48)) & m)).astype(np.int64) - IH_CENTER
    return f32_to_bf16_bits(s.astype(np.float32) * scale)


def q_rows_bf16(seed, step, seq, heads, head_dim=128):
    """bf16 bits of query rows [len(heads), head_dim] for one sequence at one step."""
    hd = np.asarray(heads, dtype=np.uint64).reshape(-1, 1)
    dim = np.arange(head_dim, dtype=np.uint64).reshape(1, -1)
    n = counter_index(TAG_Q, seq, 0, hd, 0, step, dim)
    return f32_to_bf16_bits(normal_f32_from_hash(hash64(seed, n), INV_SIGMA_F32))


def outlier_mask_bernoulli(seed, layer, head, kv, p=0.01, head_dim=128):
    """Each channel is an outlier with probability p (hash below p * 2**64)."""
    dim = np.arange(head_dim, dtype=np.uint64)
    h = hash64(seed, counter_index(TAG_OUTLIER, 0, layer, head, kv, 0, dim))
    thr = np.uint64(int(p * 2.0 ** 64))
    return h < thr


def outlier_mask_exact(seed, layer, head, kv, count=4, head_dim=128):
    """Exactly ``count`` outlier channels drawn without replacement (seeded)."""
    rng = np.random.default_rng([seed, layer, head, kv, 4242])
    m = np.zeros(head_dim, dtype=bool)
    m[rng.choice(head_dim, size=count, replace=False)] = True
    return m


def synthetic_basis(seed, layer, head, kv, head_dim=128, n_samples=8192):
    """Synthetic calibration basis U (fp32, eigenvectors as columns).

    Stand-in for the offline calibration that the pages describe (which needs
    model activations): draw a seeded Gaussian matrix, orthonormalise it
    (Householder QR) into a basis B, draw ``n_samples`` vectors
    x = sum_i sqrt(1/i) z_i b_i (spectrum 1/i), form the second moment
    C = X^T X / n (no mean removal), eigendecompose it, sort eigenvalues in
    descending order, and fix each eigenvector's sign so that its
    largest-magnitude entry is positive. Returns (U_f32, C_f64, eigvals_f64).
    """
    rng = np.random.default_rng([seed, layer, head, kv, 1717])
    B, _ = np.linalg.qr(rng.standard_normal((head_dim, head_dim)))
    Z = rng.standard_normal((n_samples, head_dim))
    spec = np.sqrt(1.0 / np.arange(1, head_dim + 1))
    X = (Z * spec) @ B.T
    C = X.T @ X / n_samples
    lam, V = np.linalg.eigh(C)
    order = np.argsort(lam)[::-1]
    lam, V = lam[order], V[:, order]
    idx = np.argmax(np.abs(V), axis=0)
    sgn = np.sign(V[idx, np.arange(head_dim)])
    V = V * sgn
    return np.ascontiguousarray(V, dtype=np.float32), C, lam


def aligned_query_rows(seed, layer, head, n, tag=0, head_dim=128):
    """bf16 bits [n, head_dim] of queries drawn with the second moment that
    synthetic_basis(seed, layer, head, kv=0) is built from: x = sum_i sqrt(1/i) z_i b_i over the
    same basis B, scaled so that E|x|^2 = head_dim. Queries for the attention-aware ablation
    (isotropic queries would make any orthogonal basis equivalent)."""
    rng = np.random.default_rng([seed, layer, head, 0, 1717])
    B, _ = np.linalg.qr(rng.standard_normal((head_dim, head_dim)))
    z = np.random.default_rng([seed, layer, head, 2929, tag]).standard_normal((n, head_dim))
    spec = np.sqrt(1.0 / np.arange(1, head_dim + 1))
    x = (z * spec) @ B.T * math.sqrt(head_dim / float(np.sum(spec * spec)))
    return f32_to_bf16_bits(x.astype(np.float32))


def config4_lengths(seed=0, batch=64, n_share=26, prefix=32768, lo=1024, hi=131072, median=16384):
    """Ragged serving batch: lognormal lengths, clipped, with a shared-prefix subset.

    Returns (lengths int64 [batch], sharer_ids sorted int64 [n_share]).
    Sharers' lengths become min(prefix + L, hi), so each sharer owns tokens past the prefix.
    """
    rng = np.random.default_rng(seed)
    L = np.exp(rng.normal(math.log(median), 1.0, size=batch))
    L = np.clip(np.rint(L), lo, hi).astype(np.int64)
    sharers = np.sort(rng.choice(batch, size=n_share, replace=False))
    L[sharers] = np.minimum(prefix + L[sharers], hi)
    return L, sharers


class Config:
    """One synthetic workload shape."""

    def __init__(self, name, batch, num_layers, num_q_heads, num_kv_heads, context,
                 group_size=128, clip=0.9, outliers="bernoulli", head_dim=128):
        self.name = name
        self.batch = batch
        self.num_layers = num_layers
        self.num_q_heads = num_q_heads
        self.num_kv_heads = num_kv_heads
        self.context = context
        self.group_size = group_size
        self.clip = clip
        self.outliers = outliers
        self.head_dim = head_dim

    def outlier_mask(self, seed, layer, head, kv):
        if self.outliers == "exact4":
            return outlier_mask_exact(seed, layer, head, kv, 4, self.head_dim)
        return outlier_mask_bernoulli(seed, layer, head, kv, 0.01, self.head_dim)


CONFIGS = {
    "tiny": Config("tiny: 1 seq x 2048, 1 layer, 4q/1kv", 1, 1, 4, 1, 2048, outliers="exact4"),
    "qwen3_8b_layer": Config("Qwen3-8B layer: 1 seq x 32768, 32q/8kv", 1, 1, 32, 8, 32768),
    "qwen3_8b_b32_100k": Config("Qwen3-8B 36 layers: 32 seqs x 100000, 32q/8kv", 32, 36, 32, 8, 100000),
    "qwen3_32b_b8_128k": Config("Qwen3-32B 64 layers: 8 seqs x 131072, 64q/8kv", 8, 64, 64, 8, 131072),
    "ragged_b64": Config("ragged serving: 64 seqs lognormal 1K-128K, 32K shared prefix, 32q/8kv",
                         64, 36, 32, 8, None),
}
