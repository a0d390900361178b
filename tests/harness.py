"""Shared GPU-vs-oracle harness: builds a pool from seeded synthetic inputs, drives it through
the C ABI (via the ctypes binding) and recomputes the same results with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workloads as W
from bit_kv_cache_paged_gb300 import Pool

# decode acceptance: |o - o_ref| <= ABS + REL * |o_ref| elementwise against the fp64 oracle
ABS_TOL = 1e-3
REL_TOL = 2e-3


def bits_to_dev(bits, shape):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).reshape(shape).cuda()


def assert_close_decode(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = ABS_TOL + REL_TOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {err.max():.3e}"
    return float(err.max())


class Case:
    """One pool plus the generator parameters that reproduce every row it holds."""

    def __init__(self, layers=1, Hq=4, Hkv=1, G=128, absorbed=False, seed=0, outliers="exact4",
                 max_seqs=4, max_len=8192, max_pages=None, clip=0.9, lloyd_a=None):
        """lloyd_a: None for the uniform levels, else [layers][Hkv][2] Lloyd-Max interior levels."""
        self.L, self.Hq, self.Hkv, self.G, self.absorbed, self.seed = layers, Hq, Hkv, G, absorbed, seed
        self.lloyd_a = None if lloyd_a is None else np.asarray(lloyd_a, dtype=np.float32)
        self.hg = Hq // Hkv
        self.clip = np.float32(clip)
        self.U = np.zeros((2, layers, Hkv, 128, 128), np.float32)
        self.mask = np.zeros((layers, Hkv, 2, 128), bool)
        for l in range(layers):
            for h in range(Hkv):
                for kv in range(2):
                    self.U[kv, l, h] = W.synthetic_basis(seed, l, h, kv)[0]
                    self.mask[l, h, kv] = (W.outlier_mask_exact(seed, l, h, kv) if outliers == "exact4"
                                           else W.outlier_mask_bernoulli(seed, l, h, kv))
        if max_pages is None:
            max_pages = max_seqs * ((max_len + 63) // 64)
        dev = torch.device("cuda")
        self.pool = Pool(layers, Hq, Hkv, max_seqs=max_seqs, max_seq_len=max_len, max_int2_pages=max_pages,
                         U_k=torch.from_numpy(self.U[0]).to(dev), U_v=torch.from_numpy(self.U[1]).to(dev),
                         clip_k=torch.full((layers, Hkv), float(clip), device=dev),
                         clip_v=torch.full((layers, Hkv), float(clip), device=dev),
                         group_size=G, v_rot_absorbed=absorbed, lloyd_max=lloyd_a is not None)
        if lloyd_a is not None:
            self.pool.set_codebook(self.lloyd_a)
        self.owner = {}   # seq -> (owner seq, shared prefix length) for prefix sharers
        self.length = {}

    def key(self, seq, pos):
        """Generator key of a position: shared-prefix positions come from the sequence shared from."""
        while seq in self.owner and pos < self.owner[seq][1]:
            seq = self.owner[seq][0]
        return seq

    def rows(self, seq, layer, head, kv, positions):
        """bf16 bits [n, 128] of K (kv=0) / V (kv=1) rows at the given positions of a sequence."""
        positions = np.asarray(positions, dtype=np.int64)
        out = np.zeros((positions.size, 128), np.uint16)
        keys = np.array([self.key(seq, int(p)) for p in positions]) if positions.size else np.zeros(0, int)
        for k in np.unique(keys):
            sel = keys == k
            out[sel] = W.kv_rows_bf16(self.seed, int(k), layer, head, kv, positions[sel], self.mask[layer, head, kv])
        return out

    def add(self, seq, share_from=-1, shared=0):
        self.pool.seq_add(seq, share_from, shared)
        if share_from >= 0:
            self.owner[seq] = (share_from, shared)
            self.length[seq] = shared
        else:
            self.length[seq] = 0

    def step(self, seq_ids, n_new):
        """One step: step_begin + append_and_demote for every layer with generator rows."""
        self.pool.step_begin(seq_ids, n_new)
        tot = int(sum(n_new))
        for l in range(self.L):
            k = np.zeros((tot, self.Hkv, 128), np.uint16)
            v = np.zeros((tot, self.Hkv, 128), np.uint16)
            r = 0
            for s, n in zip(seq_ids, n_new):
                pos = np.arange(self.length[s], self.length[s] + n)
                for h in range(self.Hkv):
                    k[r:r + n, h] = self.rows(s, l, h, 0, pos)
                    v[r:r + n, h] = self.rows(s, l, h, 1, pos)
                r += n
            kd = bits_to_dev(k, (tot, self.Hkv, 128)) if tot else None
            vd = bits_to_dev(v, (tot, self.Hkv, 128)) if tot else None
            self.pool.append_and_demote(l, kd, vd)
        for s, n in zip(seq_ids, n_new):
            self.length[s] += n

    def q_bits(self, step, seq_ids):
        return np.stack([W.q_rows_bf16(self.seed, step, s, np.arange(self.Hq)) for s in seq_ids])

    def oracle_pair(self, seq, layer, head, q_rows_f32, absorbed=None):
        """fp64 oracle output [hg, 128] for one (sequence, layer, kv head) over the GPU's packed
        INT2 cache (read back in canonical layout) and generator BF16 rows."""
        L, F, _ = self.pool.seq_info(seq)
        if F > 64:
            ck, szk, cv, szv = (t.cpu().numpy() for t in self.pool.debug_read_int2(seq, layer, head, 64, F - 64))
        else:
            ck = cv = np.zeros((0, 32), np.uint8)
            szk = szv = np.zeros((0, 128 // self.G, 2), np.float16)
        pos_b = np.r_[0:min(64, L), F:L]
        kb = W.bf16_bits_to_f32(self.rows(seq, layer, head, 0, pos_b))
        vb = W.bf16_bits_to_f32(self.rows(seq, layer, head, 1, pos_b))
        return O.decode_reference(q_rows_f32, kb, vb, O.unpack_codes(ck), szk[..., 0], szk[..., 1],
                                  O.unpack_codes(cv), szv[..., 0], szv[..., 1], self.U[0, layer, head],
                                  self.U[1, layer, head], self.G,
                                  self.absorbed if absorbed is None else absorbed,
                                  codebook=None if self.lloyd_a is None else tuple(self.lloyd_a[layer, head]))

    def decode(self, layer, step, seq_ids):
        qb = self.q_bits(step, seq_ids)
        q = bits_to_dev(qb, (len(seq_ids), self.Hq, 128))
        out = self.pool.attend(layer, q)
        self.pool.check()
        return qb, out.cpu().numpy()

    def check_decode(self, layer, step, seq_ids, heads=None):
        qb, out = self.decode(layer, step, seq_ids)
        worst = 0.0
        for i, s in enumerate(seq_ids):
            for h in (range(self.Hkv) if heads is None else heads):
                qf = W.bf16_bits_to_f32(qb[i, h * self.hg:(h + 1) * self.hg])
                ref, _ = self.oracle_pair(s, layer, h, qf)
                worst = max(worst, assert_close_decode(out[i, h * self.hg:(h + 1) * self.hg], ref,
                                                       f"seq {s} layer {layer} head {h}"))
        return worst
