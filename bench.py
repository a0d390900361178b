"""Benchmark of the OSCAR INT2 paged-KV decode hot path on GB300.

Default workload: Qwen3-8B-shaped, 36 layers, 32 query / 8 KV heads, head_dim 128, batch 32 x
context 100000 (64 BF16 sink + 99680 INT2 history + 256 BF16 recent per sequence), INT2 group 128
with fp16 scale/zero, clip 0.9, page 64, seeded synthetic K/V with 1% outlier channels x20.

One step = step_begin (1 new token per sequence) + for every layer: append_and_demote (append the
token, demote the oldest recent token into INT2), rotate_q, decode (INT2 split-K + BF16
sink/recent), merge. Inputs (cache, per-step q/k/v) are resident in HBM before timing; the cache
(66 GB) is far larger than L2, so no flush is needed between steps.

Prints one JSON line (rank 0). Besides the headline workload the line carries the other
workloads (Qwen3-32B shape at group 128 and 32, the ragged shared-prefix serving batch, the
absorbed-V and Lloyd-Max pools), a batch-1 latency case with an L2 flush between repetitions, a
read-only HBM bandwidth measurement and the CPU oracle timed in parallel on the host cores.
`--impl reference` times the CPU oracle alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: (batch, context, layers, Hq, Hkv, group)
    "qwen3_8b_b32_100k": (32, 100000, 36, 32, 8, 128),
    "qwen3_32b_b8_128k": (8, 131072, 64, 64, 8, 128),
    "qwen3_32b_b8_128k_g32": (8, 131072, 64, 64, 8, 32),
    "qwen3_8b_layer_32k": (1, 32768, 1, 32, 8, 128),
    "tiny_2k": (1, 2048, 1, 4, 1, 128),
    # ragged serving: 64 sequences with lognormal lengths 1K-128K, 26 sharing a 32768-token prefix
    # (lengths from workloads.config4_lengths; the context entry is the longest length)
    "ragged_b64": (64, 131072, 36, 32, 8, 128),
    # quantisation ablation (attention-score KL and output error against a BF16 cache)
    "ablation_b2_16k": (2, 16384, 1, 32, 8, 128),
    "ablation_b2_16k_g32": (2, 16384, 1, 32, 8, 32),
    # small cases of the same kernels for ncu captures (460 / 604 MB of INT2 pages: larger than L2)
    "prof_b8_100k_1layer": (8, 100000, 1, 32, 8, 128),
    "prof_gqa8_b8_128k_1layer": (8, 131072, 1, 64, 8, 128),
}
METRIC = "decode attn KV GB/s & tokens/s at batch32x100K vs HBM roofline; demote tok/s"
INT2_BYTES_PER_TOKEN_HEAD = {128: 72, 32: 96}
BF16_BYTES_PER_TOKEN_HEAD = 512


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="oscar", choices=["oscar", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_b32_100k", choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-bf16", action="store_true", help="skip the BF16-only cache baseline")
    ap.add_argument("--absorbed", action="store_true", help="v_rot_absorbed pool (V arrives pre-rotated)")
    ap.add_argument("--codebook", default="uniform", choices=["uniform", "lloyd_max"],
                    help="INT2 levels: uniform, or a Lloyd-Max codebook fitted per layer / KV head / K|V")
    ap.add_argument("--ablation", action="store_true",
                    help="quantisation ablation on --workload (default ablation_b2_16k): naive, clip-only, "
                         "Hadamard-only, Hadamard + clip and OSCAR rotations; prints one JSON line")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads and the latency cases (headline workload only)")
    ap.add_argument("--extra-steps", type=int, default=5, help="timed steps of each other workload")
    return ap.parse_args()


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

CALIB_SEQ = 1023   # generator sequence key of the calibration rows (workload sequences use smaller keys)
CALIB_TOKENS = 2048


def calibrate_codebook(pool, wl, seed, masks, dev):
    """Fit the Lloyd-Max interior level of every (layer, KV head, K|V) on CALIB_TOKENS generator
    rows of the calibration sequence and set the pool's codebook; returns the levels."""
    import torch

    from workloads import device as wd

    B, ctx, NL, Hq, Hkv, G = wl
    wd.build_synth()
    mdev = torch.from_numpy(masks).to(dev)
    st = torch.cuda.current_stream().cuda_stream
    rows = torch.empty((CALIB_TOKENS, Hkv, 128), dtype=torch.bfloat16, device=dev)
    a = np.ones((NL, Hkv, 2), np.float32)
    for l in range(NL):
        for kv in range(2):
            wd.fill_kv(rows, seed, CALIB_SEQ, l, kv, 0, Hkv, 0, CALIB_TOKENS, mdev[l, kv], st)
            for h in range(Hkv):
                a[l, h, kv] = pool.fit_codebook(l, h, kv, rows[:, h].contiguous(), iters=50)
    a = np.clip(a, 0.5, 1.45)
    pool.set_codebook(a)
    return a


def build_pool(wl, seed, extra_tokens, dev, lengths=None, absorbed=False, lloyd=False):
    """Pool for a workload plus its synthetic bases U and outlier masks. `lengths` (per sequence)
    sizes a ragged batch; by default every sequence has the workload's context."""
    import torch

    import workloads as W
    from bit_kv_cache_paged_gb300 import Pool

    B, ctx, NL, Hq, Hkv, G = wl
    U = np.zeros((2, NL, Hkv, 128, 128), np.float32)
    for l in range(NL):
        for h in range(Hkv):
            for kv in range(2):
                U[kv, l, h] = W.synthetic_basis(seed, l, h, kv)[0]
    if lengths is None:
        lengths = np.full(B, ctx, np.int64)
    max_len = int(max(lengths)) + extra_tokens + 64
    pages = int(sum((int(L) + extra_tokens - 320 + 63) // 64 + 1 for L in lengths))
    pool = Pool(NL, Hq, Hkv, max_seqs=B, max_seq_len=max_len, max_int2_pages=pages,
                U_k=torch.from_numpy(U[0]).to(dev), U_v=torch.from_numpy(U[1]).to(dev),
                clip_k=torch.full((NL, Hkv), 0.9, device=dev), clip_v=torch.full((NL, Hkv), 0.9, device=dev),
                group_size=G, v_rot_absorbed=absorbed, lloyd_max=lloyd)
    masks = np.zeros((NL, 2, Hkv, 128), np.uint8)
    for l in range(NL):
        for kv in range(2):
            for h in range(Hkv):
                masks[l, kv, h] = W.outlier_mask_bernoulli(seed, l, h, kv)
    return pool, U, masks


def fill_cache(pool, wl, lengths, masks, seed, dev, share=None):
    """Prefill sequence s to lengths[s] tokens: device generator -> append_and_demote (bulk demote).
    share = (owner, prefix, sharers): every sharer other than the owner takes the owner's first
    `prefix` tokens through shared page-table entries and generates only its own tokens."""
    import torch

    from workloads import device as wd

    B, ctx, NL, Hq, Hkv, G = wl
    wd.build_synth()
    mdev = torch.from_numpy(masks).to(dev)
    lengths = [int(L) for L in lengths]
    kbuf = torch.empty((max(lengths), Hkv, 128), dtype=torch.bfloat16, device=dev)
    vbuf = torch.empty_like(kbuf)
    st = torch.cuda.current_stream().cuda_stream
    demote_ms = 0.0
    rows = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    order = list(range(B))
    if share is not None:  # the owner first, so its prefix exists when the sharers attach
        order.remove(share[0])
        order.insert(0, share[0])
    for s in order:
        p0 = 0
        if share is not None and s != share[0] and s in share[2]:
            p0 = share[1]
            pool.seq_add(s, share[0], p0)
        else:
            pool.seq_add(s)
        n = lengths[s] - p0
        pool.step_begin([s], [n])
        k, v = kbuf[:n], vbuf[:n]
        for l in range(NL):
            wd.fill_kv(k, seed, s, l, 0, 0, Hkv, p0, n, mdev[l, 0], st)
            wd.fill_kv(v, seed, s, l, 1, 0, Hkv, p0, n, mdev[l, 1], st)
            e0.record()
            pool.append_and_demote(l, k, v)
            e1.record()
            e1.synchronize()
            demote_ms += e0.elapsed_time(e1)
            rows += max(0, lengths[s] - 256 - max(p0, 64)) * Hkv
    pool.check()
    return demote_ms, rows


def step_inputs(wl, L0, n_steps, seed, masks):
    """Per-step inputs (host bf16 tensors): new K/V rows [step][layer][seq][kv head][128] at
    positions L0 + step (L0 a number, or one per sequence), and q [layer][seq][q head][128]."""
    import torch

    import workloads as W

    B, ctx, NL, Hq, Hkv, G = wl
    k = np.zeros((n_steps, NL, B, Hkv, 128), np.uint16)
    v = np.zeros_like(k)
    L0s = np.broadcast_to(np.asarray(L0, np.int64), (B,))
    for l in range(NL):
        for h in range(Hkv):
            for s in range(B):
                pos = np.arange(L0s[s], L0s[s] + n_steps)
                k[:, l, s, h] = W.kv_rows_bf16(seed, s, l, h, 0, pos, masks[l, 0, h].astype(bool))
                v[:, l, s, h] = W.kv_rows_bf16(seed, s, l, h, 1, pos, masks[l, 1, h].astype(bool))
    q = np.stack([np.stack([W.q_rows_bf16(seed, l, s, np.arange(Hq)) for s in range(B)]) for l in range(NL)])
    tob = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)  # noqa: E731
    return tob(k), tob(v), tob(q)


def run_step(pool, NL, B, t, kd, vd, qd, q_rot, out):
    pool.step_begin(list(range(B)), [1] * B)
    for l in range(NL):
        pool.append_and_demote(l, kd[t, l], vd[t, l])
        pool.rotate_q(l, qd[l], q_rot)
        part = pool.decode(l, qd[l], q_rot)
        pool.merge(l, part, out[l])


def bf16_baseline(wl, args, masks, qdd, dev, n_alias=4):
    """BF16-only paged cache of the same shape: every token of every sequence in BF16 pages,
    decoded with oscar_bf16_decode. The full cache (36 layers) does not fit in HBM, so n_alias
    distinct layer caches are filled and cycled over the layers (each far larger than L2)."""
    import torch

    from bit_kv_cache_paged_gb300 import binding as Bd
    from workloads import device as wd

    B, ctx, NL, Hq, Hkv, G = wl
    n_alias = min(NL, n_alias)
    maxp = (ctx + 63) // 64
    n_pages = B * maxp
    pt = torch.arange(n_pages, dtype=torch.int32, device=dev).view(B, maxp)
    lengths = torch.full((B,), ctx, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    mdev = torch.from_numpy(masks).to(dev)
    rows = torch.empty((ctx, Hkv, 128), dtype=torch.bfloat16, device=dev)
    caches = []
    for a in range(n_alias):
        kp = torch.zeros((n_pages, Hkv, 64, 128), dtype=torch.bfloat16, device=dev)
        vp = torch.zeros_like(kp)
        for s_ in range(B):
            for kv, dst in ((0, kp), (1, vp)):
                wd.fill_kv(rows, args.seed, s_, a, kv, 0, Hkv, 0, ctx, mdev[a, kv], st)
                Bd.oscar_bf16_pack(rows, ctx, 0, Hkv, pt[s_], n_pages, dst, err, st)
        caches.append((kp, vp))
    del rows
    nb = Bd.oscar_bf16_partials_bytes(Hq, Hkv, B, ctx)
    part = torch.empty(nb, dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)

    def step():
        for l in range(NL):
            kp, vp = caches[l % n_alias]
            Bd.oscar_bf16_decode(Hq, Hkv, B, ctx, kp, vp, n_pages, pt, maxp, lengths, qdd[l], part, nb, out, err, st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    e1.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"BF16 baseline device error bits 0x{int(err.item()):x}")
    ms = e0.elapsed_time(e1) / args.steps
    step_bytes = NL * B * Hkv * ctx * BF16_BYTES_PER_TOKEN_HEAD
    del caches
    torch.cuda.empty_cache()
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(B / (ms / 1e3), 2),
            "achieved_gbs": round(step_bytes / (ms / 1e3) / 1e9, 1), "bytes_per_step": step_bytes,
            "note": f"BF16-only paged cache of the same shape, decode only (oscar_bf16_decode: split-K + merge); "
                    f"layer-aliased: {n_alias} distinct layer caches of {2 * n_pages * Hkv * 16384 / 1e9:.1f} GB "
                    f"cycled over {NL} layers (the full cache, {NL * B * Hkv * ctx * 512 / 1e9:.1f} GB, does not "
                    f"fit in HBM)"}


# rotation choice per ablation variant: "identity" = R = I (U = (H P)^T), "hp" = R = H P (U = I),
# "basis" = R = U H P with the calibration basis; then the clip ratio and whether the INT2 levels
# are a Lloyd-Max codebook fitted on calibration rows
ABLATION_VARIANTS = {"naive": ("identity", 1.0, False), "clip_only": ("identity", 0.9, False),
                     "hadamard_only": ("hp", 1.0, False), "hadamard_clip": ("hp", 0.9, False),
                     "oscar": ("basis", 0.9, False), "hadamard_clip_lloyd_max": ("hp", 0.9, True),
                     "oscar_lloyd_max": ("basis", 0.9, True)}


def hp_matrix(dev):
    """H.P as the library applies it (fp32): rows of the demote rotation of identity rows with U = I."""
    import torch

    from bit_kv_cache_paged_gb300 import Pool

    eye = torch.eye(128, device=dev)
    p = Pool(1, 4, 1, max_seqs=1, max_seq_len=1024, max_int2_pages=16, U_k=eye[None, None].contiguous(),
             U_v=eye[None, None].contiguous(), clip_k=torch.ones((1, 1), device=dev),
             clip_v=torch.ones((1, 1), device=dev))
    hp = p.debug_rotate_rows(0, 0, 0, eye.to(torch.bfloat16))
    p.close()
    return hp


def ablation_cache(wl, seed, variant_u, clip, rows_k, rows_v, dev, hp, lloyd=False):
    """Pool for one ablation variant, filled with the given device rows [B][ctx][Hkv][128]."""
    import torch

    import workloads as W
    from bit_kv_cache_paged_gb300 import Pool

    B, ctx, NL, Hq, Hkv, G = wl
    Uk = torch.empty((NL, Hkv, 128, 128), device=dev)
    Uv = torch.empty_like(Uk)
    for l in range(NL):
        for h in range(Hkv):
            for kv, U in ((0, Uk), (1, Uv)):
                if variant_u == "identity":
                    U[l, h] = hp.t()
                elif variant_u == "hp":
                    U[l, h] = torch.eye(128, device=dev)
                else:
                    U[l, h] = torch.from_numpy(W.synthetic_basis(seed, l, h, kv)[0]).to(dev)
    pool = Pool(NL, Hq, Hkv, max_seqs=B, max_seq_len=ctx + 64, max_int2_pages=B * (ctx // 64 + 1),
                U_k=Uk, U_v=Uv, clip_k=torch.full((NL, Hkv), clip, device=dev),
                clip_v=torch.full((NL, Hkv), clip, device=dev), group_size=G, lloyd_max=lloyd)
    if lloyd:
        masks = np.zeros((NL, 2, Hkv, 128), np.uint8)
        for l in range(NL):
            for kv in range(2):
                for h in range(Hkv):
                    masks[l, kv, h] = W.outlier_mask_bernoulli(seed, l, h, kv)
        calibrate_codebook(pool, wl, seed, masks, dev)
    for s_ in range(B):
        pool.seq_add(s_)
        pool.step_begin([s_], [ctx])
        for l in range(NL):
            pool.append_and_demote(l, rows_k[s_], rows_v[s_])
    pool.check()
    return pool


def ablation_inputs(wl, seed, dev):
    """Shared inputs of the ablation: device K/V rows [B][ctx][Hkv][128], aligned queries
    [B][Hq][128], the BF16-cache output o_ref (oscar_bf16_decode) and exact fp64 scores."""
    import torch

    import workloads as W
    from bit_kv_cache_paged_gb300 import binding as Bd
    from workloads import device as wd

    B, ctx, NL, Hq, Hkv, G = wl
    hg = Hq // Hkv
    wd.build_synth()
    st = torch.cuda.current_stream().cuda_stream
    masks = np.zeros((2, Hkv, 128), np.uint8)
    for kv in range(2):
        for h in range(Hkv):
            masks[kv, h] = W.outlier_mask_bernoulli(seed, 0, h, kv)
    mdev = torch.from_numpy(masks).to(dev)
    rows_k = torch.empty((B, ctx, Hkv, 128), dtype=torch.bfloat16, device=dev)
    rows_v = torch.empty_like(rows_k)
    for s_ in range(B):
        wd.fill_kv(rows_k[s_], seed, s_, 0, 0, 0, Hkv, 0, ctx, mdev[0], st)
        wd.fill_kv(rows_v[s_], seed, s_, 0, 1, 0, Hkv, 0, ctx, mdev[1], st)
    qb = np.stack([np.concatenate([W.aligned_query_rows(seed, 0, h, hg, tag=s_) for h in range(Hkv)])
                   for s_ in range(B)])
    q = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).to(dev)
    maxp = (ctx + 63) // 64
    pt = torch.arange(B * maxp, dtype=torch.int32, device=dev).view(B, maxp)
    kp = torch.zeros((B * maxp, Hkv, 64, 128), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for s_ in range(B):
        Bd.oscar_bf16_pack(rows_k[s_], ctx, 0, Hkv, pt[s_], B * maxp, kp, err, st)
        Bd.oscar_bf16_pack(rows_v[s_], ctx, 0, Hkv, pt[s_], B * maxp, vp, err, st)
    nb = Bd.oscar_bf16_partials_bytes(Hq, Hkv, B, ctx)
    part = torch.empty(nb, dtype=torch.uint8, device=dev)
    o_ref = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    lengths = torch.full((B,), ctx, dtype=torch.int32, device=dev)
    Bd.oscar_bf16_decode(Hq, Hkv, B, ctx, kp, vp, B * maxp, pt, maxp, lengths, q, part, nb, o_ref, err, st)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"BF16 reference device error bits 0x{int(err.item()):x}")
    K = rows_k.float().cpu().numpy().astype(np.float64)
    qf = W.bf16_bits_to_f32(qb).astype(np.float64)
    exact = np.empty((B, Hq, ctx))
    for s_ in range(B):
        for h in range(Hkv):
            exact[s_, h * hg:(h + 1) * hg] = qf[s_, h * hg:(h + 1) * hg] @ K[s_, :, h].T / math.sqrt(128)
    return {"rows_k": rows_k, "rows_v": rows_v, "qb": qb, "q": q, "o_ref": o_ref.double().cpu().numpy(),
            "exact": exact}


def softmax_rows(x):
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def score_kl(exact, scores):
    """Mean over rows of KL(softmax(exact) || softmax(scores)), natural log."""
    P, Q = softmax_rows(exact), softmax_rows(scores)
    return np.sum(P * (np.log(np.maximum(P, 1e-300)) - np.log(np.maximum(Q, 1e-300))), axis=-1)


def ablation_metrics(pool, wl, inp):
    """GPU side of one variant: decode output and INT2 scores from the pool; returns
    (score KL per (seq, head), output MSE per (seq, head) against o_ref, o, scores)."""
    B, ctx, NL, Hq, Hkv, G = wl
    hg = Hq // Hkv
    pool.step_begin(list(range(B)), [0] * B)
    q_rot = pool.rotate_q(0, inp["q"])
    o = pool.merge(0, pool.decode(0, inp["q"], q_rot)).double().cpu().numpy()
    pool.check()
    F = pool.seq_info(0)[1]
    sc = inp["exact"].copy()
    for s_ in range(B):
        for h in range(Hkv):
            raw = pool.debug_int2_scores(s_, 0, h, q_rot[s_, h * hg:(h + 1) * hg].contiguous(), 64, F - 64)
            sc[s_, h * hg:(h + 1) * hg, 64:F] = raw.double().cpu().numpy() / math.sqrt(128)
    mse = np.mean((o - inp["o_ref"]) ** 2, axis=-1)
    return score_kl(inp["exact"], sc), mse, o, sc


def ablation(wl, seed, dev):
    """Quantisation ablation on synthetic data (the rotation comparison of the OSCAR author
    write-up, Fig. 1 paragraph, reproduced qualitatively with this library's kernels): for each
    variant, attention-score KL(P_bf16 || P_variant) over all tokens and the output MSE
    mean((o_variant - o_bf16)^2), averaged over (sequence, query head). o_bf16 comes
    from oscar_bf16_decode over the same rows, INT2 scores from oscar_debug_int2_scores, queries
    from workloads.aligned_query_rows."""
    inp = ablation_inputs(wl, seed, dev)
    hp = hp_matrix(dev)
    out = {}
    for name, (ukind, clip, lloyd) in ABLATION_VARIANTS.items():
        pool = ablation_cache(wl, seed, ukind, clip, inp["rows_k"], inp["rows_v"], dev, hp, lloyd)
        kl, mse, _, _ = ablation_metrics(pool, wl, inp)
        out[name] = {"rotation": ukind, "clip": clip, "codebook": "lloyd_max" if lloyd else "uniform",
                     "score_kl": float(kl.mean()), "out_mse": float(mse.mean())}
        pool.close()
    return out


# ------------------------------------------------------------------------------------------------
# CPU oracle on the host cores: (sequence, KV head) units in parallel worker processes
# ------------------------------------------------------------------------------------------------

def _oracle_unit(task):
    """One (sequence, layer, KV head) unit of a decode step on the CPU oracle: the demote of the
    step's K and V row (fp64 rotation + fp32 quantiser) and the fp64 attention over the packed
    INT2 cache plus the BF16 tokens. Returns the seconds it took."""
    import oracle as O

    q, kb, vb, ck, szk, cv, szv, uk, uv, xk, xv, G = task
    t0 = time.perf_counter()
    O.encode_rows(xk, uk, 0.9, G)
    O.encode_rows(xv, uv, 0.9, G)
    O.decode_reference(q, kb, vb, O.unpack_codes(ck), szk[..., 0], szk[..., 1], O.unpack_codes(cv),
                       szv[..., 0], szv[..., 1], uk, uv, G)
    return time.perf_counter() - t0


_REF_TASK = None


def _ref_init(task):
    global _REF_TASK
    _REF_TASK = task


def _ref_unit(_):
    return _oracle_unit(_REF_TASK)


def _warm(_):
    import oracle  # noqa: F401
    import workloads  # noqa: F401
    return os.getpid()


def oracle_procs():
    return max(1, min(64, os.cpu_count() or 1))


def oracle_pool(n, initializer=None, initargs=()):
    """Worker processes for the oracle, started with `spawn` (never forked from a process that
    holds a CUDA context), each with a single-threaded BLAS so the n processes use n cores."""
    import multiprocessing as mp

    saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        return mp.get_context("spawn").Pool(n, initializer=initializer, initargs=initargs)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def cpu_model():
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_layer_oracle(pool, wl, seed, masks, U, layer=0, units=None, q_step=0):
    """Time the CPU oracle on every (sequence, KV head) unit of one layer of the current cache
    (packed INT2 pages read back from the pool, BF16 rows from the generator), in parallel worker
    processes on the host cores. Returns dict(wall_s, units, procs, unit_s_sum)."""
    import workloads as W

    B, ctx, NL, Hq, Hkv, G = wl
    hg = Hq // Hkv
    if units is None:
        units = [(s, h) for s in range(B) for h in range(Hkv)]
    tasks = []
    for s, h in units:
        L, F, _ = pool.seq_info(s)
        if F > 64:
            ck, szk, cv, szv = (x.cpu().numpy() for x in pool.debug_read_int2(s, layer, h, 64, F - 64))
        else:
            ck = cv = np.zeros((0, 32), np.uint8)
            szk = szv = np.zeros((0, 128 // G, 2), np.float16)
        pos_b = np.r_[0:min(64, L), F:L]
        mk, mv = masks[layer, 0, h].astype(bool), masks[layer, 1, h].astype(bool)
        kb = W.bf16_bits_to_f32(W.kv_rows_bf16(seed, s, layer, h, 0, pos_b, mk))
        vb = W.bf16_bits_to_f32(W.kv_rows_bf16(seed, s, layer, h, 1, pos_b, mv))
        q = W.bf16_bits_to_f32(W.q_rows_bf16(seed, q_step, s, np.arange(h * hg, (h + 1) * hg)))
        xk = W.bf16_bits_to_f32(W.kv_rows_bf16(seed, s, layer, h, 0, [max(0, F - 1)], mk))
        xv = W.bf16_bits_to_f32(W.kv_rows_bf16(seed, s, layer, h, 1, [max(0, F - 1)], mv))
        tasks.append((q, kb, vb, ck, szk, cv, szv, U[0, layer, h], U[1, layer, h], xk, xv, G))
    n = min(oracle_procs(), len(tasks))
    with oracle_pool(n) as wp:
        wp.map(_warm, range(n))  # start-up and imports outside the timed region
        t0 = time.perf_counter()
        per_unit = wp.map(_oracle_unit, tasks, chunksize=1)
        wall = time.perf_counter() - t0
    return {"wall_s": wall, "units": len(tasks), "procs": n, "unit_s_sum": float(sum(per_unit))}


def cpu_baseline_entry(cb, B, NL, Hkv, what):
    """cpu_baseline JSON object from one measured layer (all B x Hkv units), projected to NL layers."""
    step_s = cb["wall_s"] * NL
    return {"value": round(B / step_s, 6), "unit": "tokens/s", "cores": cb["procs"], "kind": "oracle",
            "cpu": cpu_model(), "measured_s": round(cb["wall_s"], 3), "measured_units": cb["units"],
            "sample": f"{what}: one full layer measured, all {cb['units']} (sequence, KV head) units (fp64 attention "
                      f"over the packed cache read back from the GPU + demote of the step's K/V rows), "
                      f"{cb['wall_s']:.2f} s wall on {cb['procs']} worker processes; "
                      + ("x%d layers projected (extrapolation)" % NL if NL > 1 else "the whole step")}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 1) for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


TRAFFIC_SOURCES = ("bit_kv_cache_paged_gb300/csrc/decode_int2.cu", "bit_kv_cache_paged_gb300/csrc/device_common.cuh",
                   "bit_kv_cache_paged_gb300/csrc/oscar_internal.h")


def kernel_source_hash():
    """sha256 (first 16 hex digits) over the INT2 decode kernel's source files."""
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_per_unit(workload):
    """DRAM bytes (read + write) per (token, KV head) of the INT2 decode kernel from the committed
    ncu capture, or None when the kernel's sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", "decode_int2_traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        if d.get("kernel_sources_sha256") != kernel_source_hash():
            return None
        return float(d["dram_bytes_per_unit"])
    except Exception:
        return None


def aggregate_replicas(elapsed_ms, world, batch, steps, device):
    """Whole-job throughput of `world` independent replicas: the slowest rank's time (max over
    ranks) and world * batch * steps tokens. Uses the default process group when world > 1."""
    if world > 1:
        import torch
        t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    return elapsed_ms, world * batch * steps / (elapsed_ms / 1e3)


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

def workload_setup(name, seed, steps, warmup, dev, absorbed=False, codebook="uniform"):
    """Pool of a workload, filled to (context - warmup - steps) tokens per sequence, plus its
    per-step inputs on the device. Returns a dict of everything the measurements use."""
    import torch

    wl = WORKLOADS[name]
    B, ctx, NL, Hq, Hkv, G = wl
    n_steps = warmup + steps
    share = None
    if name == "ragged_b64":  # per-sequence lengths and one shared prefix
        import workloads as W
        lens, sharers = W.config4_lengths(seed)
        share = (int(sharers[0]), 32768, set(int(x) for x in sharers))
        L0 = np.asarray(lens, np.int64) - n_steps
    else:
        L0 = np.full(B, ctx - n_steps, np.int64)
    pool, U, masks = build_pool(wl, seed, n_steps + 2 + 2 * steps + warmup + 2 + GRAPH_WINDOW, dev, lengths=L0 + n_steps,
                                absorbed=absorbed, lloyd=codebook == "lloyd_max")
    cb = None
    if codebook == "lloyd_max":
        a = calibrate_codebook(pool, wl, seed, masks, dev)
        cb = {"kind": "lloyd_max", "a_K_mean": round(float(a[..., 0].mean()), 4),
              "a_V_mean": round(float(a[..., 1].mean()), 4),
              "calibration": f"{CALIB_TOKENS} generator tokens per (layer, KV head, K|V)"}
    fill_ms, fill_rows = fill_cache(pool, wl, [int(x) for x in L0], masks, seed, dev, share=share)
    kd, vd, qd = step_inputs(wl, L0, n_steps, seed, masks)
    return {"name": name, "wl": wl, "pool": pool, "U": U, "masks": masks, "share": share, "L0": L0,
            "kd": kd, "vd": vd, "qd": qd, "kdd": kd.to(dev), "vdd": vd.to(dev), "qdd": qd.to(dev),
            "q_rot": torch.empty((B, Hq, 128), dtype=torch.float32, device=dev),
            "out": torch.empty((NL, B, Hq, 128), dtype=torch.float32, device=dev),
            "fill_ms": fill_ms, "fill_rows": fill_rows, "codebook": cb, "n_steps": n_steps,
            "steps": steps, "warmup": warmup}


GRAPH_WINDOW = 64


def measure_steps(ws, world, dev, breakdown=True, graph=True, window=False):
    """Warm-up, then the timed per-layer-call steps (events around every INT2 decode launch: the
    roofline's timed region), the per-kernel breakdown, and the same steps as one CUDA graph each.
    Returns a dict of raw numbers."""
    import torch

    pool, (B, ctx, NL, Hq, Hkv, G) = ws["pool"], ws["wl"]
    kdd, vdd, qdd, q_rot, out = ws["kdd"], ws["vdd"], ws["qdd"], ws["q_rot"], ws["out"]
    steps, warmup, n_steps = ws["steps"], ws["warmup"], ws["n_steps"]
    stream = torch.cuda.current_stream()
    for t in range(warmup):
        run_step(pool, NL, B, t, kdd, vdd, qdd, q_rot, out)
    pool.check()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    pool.timing_enable(["decode_int2"])  # events around the dominant kernel only
    n0 = pool.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    int2_units = 0
    torch.cuda.nvtx.range_push("timed")
    torch.cuda.profiler.start()  # no-op unless a profiler runs with --profile-from-start off
    ev0.record(stream)
    for t in range(warmup, n_steps):
        run_step(pool, NL, B, t, kdd, vdd, qdd, q_rot, out)
        int2_units += sum(pool.seq_info(s)[1] - 64 for s in range(B)) * Hkv * NL
    ev1.record(stream)
    torch.cuda.profiler.stop()
    torch.cuda.nvtx.range_pop()
    ev1.synchronize()
    r = {"layer_elapsed_ms": ev0.elapsed_time(ev1), "layer_launches": pool.launch_count() - n0,
         "int2_units": int2_units}
    r["ktimes"] = pool.timing_read()
    pool.timing_enable(False)
    pool.check()
    r["kbreak"] = None
    if breakdown:  # two extra steps (outside the timed region) with every launch timed
        pool.timing_enable(True)
        for _ in range(2):  # re-appends the last timed step's rows (values do not affect timing)
            run_step(pool, NL, B, n_steps - 1, kdd, vdd, qdd, q_rot, out)
        r["kbreak"] = pool.timing_read()
        pool.timing_enable(False)
    r["graph_ms"] = None
    r["window"] = None
    if graph:
        # the same steps as one CUDA graph launch each (all layers' kernels); the appended rows
        # repeat the last timed step's (values do not affect timing), so the graph's pointers stay
        kg, vg = kdd[n_steps - 1], vdd[n_steps - 1]
        for _ in range(warmup):
            pool.step_begin(list(range(B)), [1] * B)
            pool.step_graph(kg, vg, qdd, q_rot, out)
        pool.check()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gn0 = pool.launch_count()
        g0.record(stream)
        for _ in range(steps):
            pool.step_begin(list(range(B)), [1] * B)
            pool.step_graph(kg, vg, qdd, q_rot, out)
        g1.record(stream)
        g1.synchronize()
        r["graph_launches"] = pool.launch_count() - gn0
        pool.check()
        r["graph_ms"] = g0.elapsed_time(g1)
        if window:
            # GRAPH_WINDOW more graph steps: every sequence starts a new INT2 page on the way; the
            # graph is relaunched, not recorded again
            c0 = pool.graph_captures()
            w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            p0 = [pool.seq_info(s)[2] for s in range(B)]
            w0.record(stream)
            for _ in range(GRAPH_WINDOW):
                pool.step_begin(list(range(B)), [1] * B)
                pool.step_graph(kg, vg, qdd, q_rot, out)
            w1.record(stream)
            w1.synchronize()
            pool.check()
            wms = w0.elapsed_time(w1)
            r["window"] = {"steps": GRAPH_WINDOW, "ms_per_step": round(wms / GRAPH_WINDOW, 4),
                           "tokens_per_s": round(B * GRAPH_WINDOW / (wms / 1e3), 2),
                           "graph_recordings": pool.graph_captures() - c0,
                           "sequences_with_a_new_int2_page": sum(pool.seq_info(s)[2] > p for s, p in zip(range(B), p0)),
                           "note": "one CUDA graph per step over a window in which every sequence starts a new INT2 "
                                   "page; graph_recordings counts re-captures inside the window"}
    return r


def decode_roofline(r, G, peak, read_peak):
    d_ms, d_n = r["ktimes"]["decode_int2"]
    int2_bytes = r["int2_units"] * INT2_BYTES_PER_TOKEN_HEAD[G]
    gbs = int2_bytes / (d_ms / 1e3) / 1e9 if d_ms > 0 else None
    return {"achieved": round(gbs, 1) if gbs else None, "frac": round(gbs / peak, 4) if gbs else None,
            "frac_of_read_peak": round(gbs / read_peak, 4) if (gbs and read_peak) else None,
            "int2_bytes": int2_bytes, "launches": d_n, "ms": d_ms}


def extra_workload(name, args, dev, peak, read_peak, absorbed=False, codebook="uniform", cpu=False):
    """A workload other than the headline, in the same measurement: tokens/s as one CUDA graph per
    step, the INT2 decode kernel's GB/s and roofline fraction, the per-kernel split of a step and
    (cpu=True) the CPU oracle on one full layer."""
    import torch

    t_start = time.perf_counter()
    ws = workload_setup(name, args.seed, args.extra_steps, 3, dev, absorbed=absorbed, codebook=codebook)
    B, ctx, NL, Hq, Hkv, G = ws["wl"]
    r = measure_steps(ws, 1, dev)
    rl = decode_roofline(r, G, peak, read_peak)
    pool = ws["pool"]
    int2_tok = sum(pool.seq_info(s)[1] - 64 for s in range(B))
    share = ws["share"]
    shared_tok = (len(share[2]) - 1) * (share[1] - 64) if share is not None else 0
    res = {"workload": name, "batch": B, "context": ctx, "layers": NL, "q_heads": Hq, "kv_heads": Hkv,
           "group_size": G, "v_rot_absorbed": absorbed, "codebook": ws["codebook"] or "uniform",
           "steps": args.extra_steps, "warmup": 3,
           "tokens_per_s": round(B * args.extra_steps / (r["graph_ms"] / 1e3), 2),
           "ms_per_step": round(r["graph_ms"] / args.extra_steps, 4),
           "decode_int2": {"gbs": rl["achieved"], "frac": rl["frac"], "frac_of_read_peak": rl["frac_of_read_peak"],
                           "ms_per_step": round(rl["ms"] / args.extra_steps, 4)},
           "kernels_ms_per_step": {k: round(v[0] / 2, 4) for k, v in r["kbreak"].items()},
           "int2_gb_logical": round(int2_tok * Hkv * NL * INT2_BYTES_PER_TOKEN_HEAD[G] / 1e9, 2),
           "int2_gb_unique": round((int2_tok - shared_tok) * Hkv * NL * INT2_BYTES_PER_TOKEN_HEAD[G] / 1e9, 2)}
    if share is not None:
        res["roofline_bytes"] = "logical (each sharer reads the shared pages)"
        res["lengths"] = "workloads.config4_lengths: 64 lognormal lengths, 26 share a 32768-token prefix"
    if cpu:
        cb = cpu_layer_oracle(pool, ws["wl"], args.seed, ws["masks"], ws["U"])
        res["cpu_baseline"] = cpu_baseline_entry(cb, B, NL, Hkv, name)
    pool.close()
    del ws
    torch.cuda.empty_cache()
    res["wall_s"] = round(time.perf_counter() - t_start, 1)
    return res


def flush_l2(buf):
    buf.fill_(1)


def latency_case(name, args, dev, reps=50):
    """Latency of one decode step of a small workload whose cache fits in L2: before every
    repetition a 256 MiB buffer (twice the L2) is written, so each step starts cold. Reports the
    device time of the step as one graph launch, each kernel's device time (events around every
    launch, per-layer calls), and the INT2 decode's split count (workers per (sequence, KV head))."""
    import torch

    ws = workload_setup(name, args.seed, 2 * reps + 4, 3, dev)
    pool, (B, ctx, NL, Hq, Hkv, G) = ws["pool"], ws["wl"]
    kdd, vdd, qdd, q_rot, out = ws["kdd"], ws["vdd"], ws["qdd"], ws["q_rot"], ws["out"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for t in range(3):
        run_step(pool, NL, B, t, kdd, vdd, qdd, q_rot, out)
    pool.check()
    # per-kernel device times, every launch bracketed by events
    pool.timing_enable(True)
    t = 3
    for _ in range(reps):
        flush_l2(flush)
        run_step(pool, NL, B, t, kdd, vdd, qdd, q_rot, out)
        t += 1
    kt = pool.timing_read()
    pool.timing_enable(False)
    n_pairs = B * Hkv
    workers = pool.int2_workers()
    # the step as one graph launch (host step_begin outside the events)
    kg, vg = kdd[t], vdd[t]
    times = []
    for i in range(reps + 3):
        flush_l2(flush)
        pool.step_begin(list(range(B)), [1] * B)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pool.step_graph(kg, vg, qdd, q_rot, out)
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e3)
    pool.check()
    res = {"workload": name, "batch": B, "context": ctx, "layers": NL, "q_heads": Hq, "kv_heads": Hkv,
           "l2_flush": "256 MiB written before every repetition", "reps": reps,
           "graph_us_per_step": {"median": round(float(np.median(times)), 2), "min": round(float(np.min(times)), 2)},
           "kernel_us": {k: round(v[0] / max(1, v[1]) * 1e3, 2) for k, v in kt.items() if v[1]},
           "int2_workers": int(workers), "int2_workers_per_kv_head": round(workers / n_pairs, 2),
           "int2_pages_per_kv_head": int((pool.seq_info(0)[1] - 64 + 63) // 64)}
    cb = cpu_layer_oracle(pool, ws["wl"], args.seed, ws["masks"], ws["U"])
    res["cpu_baseline"] = cpu_baseline_entry(cb, B, NL, Hkv, name)
    pool.close()
    del ws, flush
    torch.cuda.empty_cache()
    return res


def gpu_arm(args, rank, world):
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    import __graft_entry__ as ge
    if rank == 0:
        ge.build()
    if world > 1:
        torch.distributed.barrier()
    ge.build()
    from workloads import device as wd

    peaks = load_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    read_peak = wd.read_stream_gbs(dev)

    ws = workload_setup(args.workload, args.seed, args.steps, args.warmup, dev, absorbed=args.absorbed,
                        codebook=args.codebook)
    wl, pool, U, masks, share = ws["wl"], ws["pool"], ws["U"], ws["masks"], ws["share"]
    B, ctx, NL, Hq, Hkv, G = wl
    kdd, vdd, qdd, q_rot, out = ws["kdd"], ws["vdd"], ws["qdd"], ws["q_rot"], ws["out"]
    n_steps = ws["n_steps"]
    stream = torch.cuda.current_stream()

    clocks = ClockSampler(dev.index)
    clocks.start()
    r = measure_steps(ws, world, dev, graph=not args.no_graph, window=True)
    clk = clocks.stop()
    layer_ms, layer_tok_s = aggregate_replicas(r["layer_elapsed_ms"], world, B, args.steps, dev)
    per_layer = {"ms_per_step": round(layer_ms / args.steps, 4), "tokens_per_s": round(layer_tok_s, 2),
                 "note": "the same steps as per-layer calls (append_and_demote, rotate_q, decode, merge) with "
                         "CUDA events around every decode_int2 launch: the roofline's timed region"}
    if r["graph_ms"] is not None:
        elapsed_ms, tok_s = aggregate_replicas(r["graph_ms"], world, B, args.steps, dev)
        launches = r["graph_launches"]
        path = ("oscar_step_graph: one CUDA graph launch per step holding every layer's append_and_demote, "
                "rotate_q, decode and merge; host step_begin included")
    else:
        elapsed_ms, tok_s, launches = layer_ms, layer_tok_s, r["layer_launches"]
        path = "per-layer calls"
    ms_step = elapsed_ms / args.steps
    rl = decode_roofline(r, G, peak, read_peak)
    d_ms, d_n = rl["ms"], rl["launches"]
    int2_bytes = rl["int2_bytes"]
    step_bytes = (int2_bytes + args.steps * NL * B * Hkv * 320 * BF16_BYTES_PER_TOKEN_HEAD)
    tpu = traffic_per_unit(args.workload)
    traffic = tpu * (r["int2_units"] / d_n) if (tpu is not None and d_n) else None
    kbreak = r["kbreak"]

    # e2e: host buffers through the C ABI: every step copies its inputs in from pinned host memory
    # and its outputs back. The copies run on a second stream through device staging buffers, so
    # they overlap the previous / next step's compute; the step graph keeps its fixed buffers,
    # filled and drained by device-to-device copies on the compute stream.
    e2e = None
    if not args.no_e2e:
        extra = args.steps
        hk, hv, hq = step_inputs(wl, ws["L0"] + n_steps + 2, extra, args.seed, masks)
        hk, hv, hq = hk.pin_memory(), hv.pin_memory(), ws["qd"].pin_memory()
        hout = torch.empty((extra,) + tuple(out.shape), dtype=torch.float32).pin_memory()
        dk = torch.empty(hk.shape[1:], dtype=torch.bfloat16, device=dev)
        dv = torch.empty_like(dk)
        dq = torch.empty(hq.shape, dtype=torch.bfloat16, device=dev)
        stage = [(torch.empty_like(dk), torch.empty_like(dv), torch.empty_like(dq), torch.empty_like(out))
                 for _ in range(2)]
        cstream = torch.cuda.Stream(device=dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        in_free = [torch.cuda.Event() for _ in range(2)]
        out_ready = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]
        for b in range(2):
            in_free[b].record(stream)
            out_free[b].record(stream)

        def copy_in(t):
            b = t & 1
            with torch.cuda.stream(cstream):
                cstream.wait_event(in_free[b])
                stage[b][0].copy_(hk[t], non_blocking=True)
                stage[b][1].copy_(hv[t], non_blocking=True)
                stage[b][2].copy_(hq, non_blocking=True)
                in_ready[b].record(cstream)

        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_in(0)
        for t in range(extra):
            b = t & 1
            if t + 1 < extra:
                copy_in(t + 1)
            stream.wait_event(in_ready[b])
            dk.copy_(stage[b][0], non_blocking=True)
            dv.copy_(stage[b][1], non_blocking=True)
            dq.copy_(stage[b][2], non_blocking=True)
            in_free[b].record(stream)
            pool.step_begin(list(range(B)), [1] * B)
            if args.no_graph:
                for l in range(NL):
                    pool.append_and_demote(l, dk[l], dv[l])
                    pool.rotate_q(l, dq[l], q_rot)
                    part = pool.decode(l, dq[l], q_rot)
                    pool.merge(l, part, out[l])
            else:
                pool.step_graph(dk, dv, dq, q_rot, out)
            stream.wait_event(out_free[b])
            stage[b][3].copy_(out, non_blocking=True)
            out_ready[b].record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(out_ready[b])
                hout[t].copy_(stage[b][3], non_blocking=True)
                out_free[b].record(cstream)
        stream.wait_stream(cstream)
        e1.record(stream)
        e1.synchronize()
        e_ms = e0.elapsed_time(e1)
        pool.check()
        h2d = (hk[0].numel() + hv[0].numel() + hq.numel()) * 2
        e2e = {"value": round(world * B * extra / (e_ms / 1e3), 2), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hout[0].numel() * 4),
               "note": "pinned host inputs in and every layer's output out each step; the copies overlap "
                       "compute on a second stream through device staging buffers"}

    bf16 = None
    if not args.no_bf16:
        bf16 = bf16_baseline(wl, args, masks, qdd, dev)
        bf16["frac"] = round(bf16["achieved_gbs"] / peak, 4)
        bf16["int2_path_speedup"] = round(tok_s / world / bf16["tokens_per_s"], 3)

    # INT2 cache size: logical (every sequence's history) and unique (a shared prefix counted once)
    int2_tok = sum(pool.seq_info(s)[1] - 64 for s in range(B))
    int2_gb = int2_tok * Hkv * NL * INT2_BYTES_PER_TOKEN_HEAD[G] / 1e9
    shared_tok = (len(share[2]) - 1) * (share[1] - 64) if share is not None else 0
    int2_gb_unique = (int2_tok - shared_tok) * Hkv * NL * INT2_BYTES_PER_TOKEN_HEAD[G] / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cb = cpu_layer_oracle(pool, wl, args.seed, masks, U)
        cpu = cpu_baseline_entry(cb, B, NL, Hkv, args.workload)
    fill_ms, fill_rows = ws["fill_ms"], ws["fill_rows"]
    codebook = ws["codebook"]
    pool.close()
    del ws, kdd, vdd, qdd, q_rot, out
    torch.cuda.empty_cache()

    res = {
        "metric": METRIC, "value": round(tok_s, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int2-kv f16-mma f32-acc", "data": "synthetic",
        "config": {"workload": args.workload, "batch": B, "context": ctx, "layers": NL, "q_heads": Hq,
                   "kv_heads": Hkv, "head_dim": 128, "group_size": G, "page": 64, "sink": 64, "recent": 256,
                   "clip": 0.9, "v_rot_absorbed": bool(args.absorbed), "codebook": codebook or "uniform",
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (INT2 cache %.1f GB)" % int2_gb,
                   **({"int2_gb_logical": round(int2_gb, 2), "int2_gb_unique": round(int2_gb_unique, 2),
                       "lengths": "workloads.config4_lengths: 64 lognormal lengths, 26 share a 32768-token prefix",
                       "roofline_bytes": "logical (each sharer reads the shared pages)"} if share is not None else {})},
        "roofline": {"kernel": "decode_int2", "bound": "hbm", "achieved": rl["achieved"],
                     "peak": peak, "unit": "GB/s", "frac": rl["frac"],
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks else "fallback 6800 GB/s (of fallback)",
                     "read_peak": round(read_peak, 1), "frac_of_read_peak": rl["frac_of_read_peak"],
                     "read_peak_source": "this run: read-only streaming kernel over 8 GiB, best of 5 (CUDA events)",
                     "traffic": traffic, "algorithmic_bytes_per_launch": int(int2_bytes / max(1, d_n)),
                     "avg_launch_ms": round(d_ms / max(1, d_n), 5)},
        "step_gbs": round(step_bytes / (elapsed_ms / 1e3) / 1e9, 1),
        "kernels_ms_per_step": {k: round(v[0] / 2, 4) for k, v in kbreak.items()},
        "demote": {"bulk_rows_per_s": round(fill_rows * 2 / (fill_ms / 1e3), 1),
                   "bulk_gbs": round(fill_rows * 2 * 292 / (fill_ms / 1e3) / 1e9, 1),
                   "bulk_frac": round(fill_rows * 2 * 292 / (fill_ms / 1e3) / 1e9 / peak, 4),
                   "bulk_note": "prefill demote (K and V rows, all layers) timed per launch with CUDA events; "
                                "292 B per row (256 B bf16 read, 32 B codes + 4 B scale/zero written)",
                   "step_rows_per_s": round(B * Hkv * 2 * NL * 2 / (kbreak["demote"][0] / 1e3), 1)
                   if kbreak["demote"][0] > 0 else None},
        "path": path, "per_layer_calls": per_layer, "graph_window": r["window"], "bf16_baseline": bf16, "e2e": e2e, "gpu_launches": int(launches),
        "clocks": clk, "cpu_baseline": cpu,
    }
    if rank == 0 and world == 1 and not args.no_extra:
        extras = {}
        for key, (name, kw) in EXTRA_WORKLOADS.items():
            extras[key] = extra_workload(name, args, dev, peak, read_peak, **kw)
        res["extra_workloads"] = extras
        res["latency"] = {name: latency_case(name, args, dev) for name in LATENCY_WORKLOADS}
    if rank == 0:
        print(json.dumps(res), flush=True)


# workloads measured beside the headline: key -> (workload, options)
EXTRA_WORKLOADS = {
    "qwen3_32b_b8_128k": ("qwen3_32b_b8_128k", {"cpu": True}),
    "qwen3_32b_b8_128k_g32": ("qwen3_32b_b8_128k_g32", {"cpu": True}),
    "ragged_b64": ("ragged_b64", {"cpu": True}),
    "qwen3_8b_b32_100k_absorbed": ("qwen3_8b_b32_100k", {"absorbed": True}),
    "qwen3_8b_b32_100k_lloyd_max": ("qwen3_8b_b32_100k", {"codebook": "lloyd_max"}),
}
LATENCY_WORKLOADS = ("qwen3_8b_layer_32k", "tiny_2k")


# ------------------------------------------------------------------------------------------------
# Reference arm: the CPU oracle
# ------------------------------------------------------------------------------------------------

def reference_arm(args, rank, world):
    """The CPU oracle on the host cores: every step runs one bounded sample of the workload's decode
    step, one (sequence, KV head) unit per worker process at full context (the oracle's demote of
    the step's K and V row and its fp64 attention over an oracle-encoded INT2 cache), all in
    parallel. ms_per_step is the measured wall time of that sample; value and
    projected_ms_per_step scale it to the whole step (batch x KV heads x layers units)."""
    if rank != 0:
        return
    import oracle as O
    import workloads as W

    wl = WORKLOADS[args.workload]
    B, ctx, NL, Hq, Hkv, G = wl
    hg = Hq // Hkv
    seed = args.seed
    L = ctx
    F = L - 256
    s, l, h = 0, 0, 0
    mk = W.outlier_mask_bernoulli(seed, l, h, 0)
    mv = W.outlier_mask_bernoulli(seed, l, h, 1)
    Uk = W.synthetic_basis(seed, l, h, 0)[0]
    Uv = W.synthetic_basis(seed, l, h, 1)[0]
    pos = np.arange(64, F)
    enc_k = O.encode_rows(W.bf16_bits_to_f32(W.kv_rows_bf16(seed, s, l, h, 0, pos, mk)), Uk, 0.9, G)
    enc_v = O.encode_rows(W.bf16_bits_to_f32(W.kv_rows_bf16(seed, s, l, h, 1, pos, mv)), Uv, 0.9, G)
    pos_b = np.r_[0:64, F:L]
    kb = W.bf16_bits_to_f32(W.kv_rows_bf16(seed, s, l, h, 0, pos_b, mk))
    vb = W.bf16_bits_to_f32(W.kv_rows_bf16(seed, s, l, h, 1, pos_b, mv))
    q = W.bf16_bits_to_f32(W.q_rows_bf16(seed, 0, s, np.arange(hg)))
    task = (q, kb, vb, O.pack_codes(enc_k["codes"]), np.stack([enc_k["s16"], enc_k["z16"]], -1),
            O.pack_codes(enc_v["codes"]), np.stack([enc_v["s16"], enc_v["z16"]], -1), Uk, Uv, kb[-1:], vb[-1:], G)
    units_full = B * Hkv * NL
    n = min(oracle_procs(), units_full)
    with oracle_pool(n, initializer=_ref_init, initargs=(task,)) as wp:
        for _ in range(args.warmup):
            wp.map(_ref_unit, range(n), chunksize=1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            wp.map(_ref_unit, range(n), chunksize=1)
        dt = (time.perf_counter() - t0) / args.steps
    step_s = dt * units_full / n
    val = B / step_s
    res = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 1),
           "projected_ms_per_step": round(step_s * 1e3, 1),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": args.workload, "batch": B, "context": ctx, "layers": NL, "q_heads": Hq,
                      "kv_heads": Hkv, "head_dim": 128, "group_size": G, "page": 64, "sink": 64, "recent": 256,
                      "clip": 0.9, "v_rot_absorbed": bool(args.absorbed), "codebook": "uniform",
                      "parallelism": f"replicas x{world}"},
           "cpu_baseline": {"value": round(val, 6), "unit": "tokens/s", "cores": n, "kind": "oracle", "cpu": cpu_model(),
                            "sample": f"each step: {n} (sequence, KV head) units at context {ctx} in parallel on {n} "
                                      f"worker processes (fp64 attention over an oracle-encoded INT2 cache + demote of "
                                      f"1 K and 1 V row each), measured {dt:.3f} s wall per step (ms_per_step); a full "
                                      f"decode step is {units_full} units: projected_ms_per_step"},
           "e2e": {"value": round(val, 6), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "oscar":
        import torch
        torch.distributed.init_process_group("nccl")
    if args.ablation:
        import torch
        if args.workload == "qwen3_8b_b32_100k":
            args.workload = "ablation_b2_16k"
        torch.cuda.set_device(0)
        import __graft_entry__ as ge
        ge.build()
        res = ablation(WORKLOADS[args.workload], args.seed, torch.device("cuda", 0))
        print(json.dumps({"ablation": res, "workload": args.workload, "data": "synthetic",
                          "queries": "aligned to the calibration basis (workloads.aligned_query_rows)"}), flush=True)
        return
    if args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        gpu_arm(args, rank, world)
    if world > 1 and args.impl == "oscar":
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
