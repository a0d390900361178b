"""Quantisation ablation diagnostics against the oracle.

The diagnostics (bench.py --ablation) compare five rotation/clipping variants by attention-score
KL and relative output error against a BF16 cache, computed from this library's kernels. Here the
same numbers are recomputed from the oracle on the GPU's packed cache: INT2 scores from the
oracle's dequantisation and rotation, outputs from decode_reference, the BF16 reference from plain
fp64 attention, and the KL written out independently."""
import math

import numpy as np
import pytest
import torch

import bench
import oracle as O
import workloads as W
from harness import assert_close_decode

WL = (1, 4096, 1, 4, 1, 128)  # 1 sequence x 4096 tokens, 1 layer, 4 q / 1 KV head, group 128


def _kl(p_logits, q_logits):
    p = np.exp(p_logits - p_logits.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    q = np.exp(q_logits - q_logits.max(axis=-1, keepdims=True))
    q /= q.sum(axis=-1, keepdims=True)
    return np.sum(p * np.log(p / q), axis=-1)


def _pool_codebook(pool, wl, dev):
    """The (a_K, a_V) a Lloyd-Max ablation pool was calibrated with: refit on the same calibration
    rows (the fit is deterministic) and check it against the oracle's fit on the GPU's rotated rows."""
    from workloads import device as wd
    B, ctx, NL, Hq, Hkv, G = wl
    masks = torch.from_numpy(np.stack([np.stack([W.outlier_mask_bernoulli(0, 0, h, kv) for h in range(Hkv)])
                                       for kv in range(2)]).astype(np.uint8)).to(dev)
    rows = torch.empty((bench.CALIB_TOKENS, Hkv, 128), dtype=torch.bfloat16, device=dev)
    out = []
    for kv in range(2):
        wd.fill_kv(rows, 0, bench.CALIB_SEQ, 0, kv, 0, Hkv, 0, bench.CALIB_TOKENS, masks[kv],
                   torch.cuda.current_stream().cuda_stream)
        x = rows[:, 0].contiguous()
        a = pool.fit_codebook(0, 0, kv, x, iters=50)
        rot32 = pool.debug_rotate_rows(0, 0, kv, x).cpu().numpy()
        a_or = O.lloyd_fit(O.normalized_rows(rot32, np.float32(0.9), G), iters=50)
        assert abs(a - np.float32(a_or)) <= 1e-6
        out.append(float(np.clip(np.float32(a), 0.5, 1.45)))
    return out


def test_score_kl_closed_form():
    """bench.score_kl against KL of two-point distributions in closed form, and KL(P||P) = 0."""
    a = np.array([[0.0, math.log(3.0)]])  # P = (1/4, 3/4)
    b = np.array([[0.0, 0.0]])            # Q = (1/2, 1/2)
    want = 0.25 * math.log(0.5) + 0.75 * math.log(1.5)
    assert abs(bench.score_kl(a, b)[0] - want) < 1e-12
    assert abs(bench.score_kl(a, a)[0]) < 1e-15


@pytest.mark.gpu
def test_ablation_metrics_match_oracle():
    import __graft_entry__ as g
    g.build()
    dev = torch.device("cuda")
    B, ctx, NL, Hq, Hkv, G = WL
    inp = bench.ablation_inputs(WL, 0, dev)
    hp = bench.hp_matrix(dev)
    assert np.abs(hp.cpu().numpy() - O.rotation_matrix(np.eye(128))).max() < 1e-6  # H.P as the oracle has it
    K = inp["rows_k"][0, :, 0].float().cpu().numpy().astype(np.float64)
    V = inp["rows_v"][0, :, 0].float().cpu().numpy().astype(np.float64)
    qf = W.bf16_bits_to_f32(inp["qb"][0]).astype(np.float64)
    o_bf16, _ = O.attention(qf, K, V)
    assert_close_decode(inp["o_ref"][0], o_bf16, "BF16 reference")
    exact = qf @ K.T / math.sqrt(128)
    kls = {}
    for name, (ukind, clip, lloyd) in bench.ABLATION_VARIANTS.items():
        pool = bench.ablation_cache(WL, 0, ukind, clip, inp["rows_k"], inp["rows_v"], dev, hp, lloyd)
        cb = None
        if lloyd:  # the codebook the pool was given, read back through the fit on the same rows
            cb = tuple(_pool_codebook(pool, WL, dev))
        kl, mse, o, sc = bench.ablation_metrics(pool, WL, inp)
        U = {0: None, 1: None}
        for kv in (0, 1):
            if ukind == "identity":
                U[kv] = hp.t().cpu().numpy()
            elif ukind == "hp":
                U[kv] = np.eye(128, dtype=np.float32)
            else:
                U[kv] = W.synthetic_basis(0, 0, 0, kv)[0]
        L, F, _ = pool.seq_info(0)
        ck, szk, cv, szv = (t.cpu().numpy() for t in pool.debug_read_int2(0, 0, 0, 64, F - 64))
        k_hat = (O.dequantize(O.unpack_codes(ck), szk[..., 0], szk[..., 1], G) if cb is None else
                 O.dequantize_lloyd(O.unpack_codes(ck), szk[..., 0], szk[..., 1], G, cb[0]))
        q_rot = qf @ O.rotation_matrix(U[0])
        sc_or = exact.copy()
        sc_or[:, 64:F] = q_rot @ k_hat.T / math.sqrt(128)
        np.testing.assert_allclose(sc[0], sc_or, atol=2e-4, rtol=1e-4, err_msg=f"{name} scores")
        kl_or = _kl(exact, sc_or)
        np.testing.assert_allclose(kl[0], kl_or, rtol=2e-3, atol=1e-7, err_msg=f"{name} KL")
        pos_b = np.r_[0:64, F:L]
        o_or, _ = O.decode_reference(qf, K[pos_b], V[pos_b], O.unpack_codes(ck), szk[..., 0], szk[..., 1],
                                     O.unpack_codes(cv), szv[..., 0], szv[..., 1], U[0], U[1], G, codebook=cb)
        assert_close_decode(o[0], o_or, f"{name} decode")
        mse_or = np.mean((o_or - o_bf16) ** 2, axis=-1)
        np.testing.assert_allclose(mse[0], mse_or, rtol=2e-2, atol=1e-9, err_msg=f"{name} output MSE")
        kls[name] = float(kl_or.mean())
        pool.close()
    # channel outliers x20 dominate the group range without a rotation
    assert kls["naive"] > kls["hadamard_only"]
