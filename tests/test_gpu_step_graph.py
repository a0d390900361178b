"""oscar_step_graph (one CUDA graph per decode step) against the same step made of per-layer calls.

Two pools built from the same seeded inputs go through the same steps: one through
append_and_demote / rotate_q / decode / merge layer by layer, the other through the graph. Outputs
must be bit-identical (same kernels, same inputs). The steps cross INT2 page boundaries, change the
batch and append several tokens at once, so the graph is both relaunched and re-captured."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import Case, assert_close_decode, bits_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__ as g
    g.build()


def _inputs(c, ids, n_new, step):
    """k/v bf16 [layers][Σn_new][Hkv][128] for the next tokens of ids, q [layers][n][Hq][128]."""
    tot = int(sum(n_new))
    k = np.zeros((c.L, tot, c.Hkv, 128), np.uint16)
    v = np.zeros_like(k)
    for l in range(c.L):
        r = 0
        for s, n in zip(ids, n_new):
            pos = np.arange(c.length[s], c.length[s] + n)
            for h in range(c.Hkv):
                k[l, r:r + n, h] = c.rows(s, l, h, 0, pos)
                v[l, r:r + n, h] = c.rows(s, l, h, 1, pos)
            r += n
    q = np.stack([np.stack([W.q_rows_bf16(c.seed, 1000 * step + l, s, np.arange(c.Hq)) for s in ids])
                  for l in range(c.L)])
    return (bits_to_dev(k, k.shape), bits_to_dev(v, v.shape), bits_to_dev(q, q.shape), q)


def test_step_graph_equals_per_layer_calls():
    lengths = [1000, 2047, 300]
    ids = [0, 1, 2]
    a = Case(layers=2, Hq=8, Hkv=2, max_seqs=3, max_len=3000)
    b = Case(layers=2, Hq=8, Hkv=2, max_seqs=3, max_len=3000)
    for c in (a, b):
        for s in ids:
            c.add(s)
        c.step(ids, lengths)
    plan = [(ids, [1, 1, 1])] * 70 + [([2, 0], [5, 1]), (ids, [1, 1, 1]), ([1], [1]), (ids, [1, 1, 1])]
    bufs = {}
    for step, (sids, n_new) in enumerate(plan):
        k, v, q, qb = _inputs(a, sids, n_new, step)
        # per-layer calls
        a.pool.step_begin(sids, n_new)
        a0 = a.pool.launch_count()
        out_a = []
        for l in range(a.L):
            a.pool.append_and_demote(l, k[l], v[l])
            q_rot = a.pool.rotate_q(l, q[l])
            out_a.append(a.pool.merge(l, a.pool.decode(l, q[l], q_rot)).clone())
        a_launched = a.pool.launch_count() - a0  # the graph holds the same kernels
        # one graph launch; inputs staged in persistent buffers so that steps of the same shape
        # relaunch the graph instead of capturing a new one
        b.pool.step_begin(sids, n_new)
        shape = (k.shape[1], len(sids))
        if shape not in bufs:
            bufs[shape] = (torch.empty_like(k), torch.empty_like(v), torch.empty_like(q),
                           torch.empty((len(sids), b.Hq, 128), dtype=torch.float32, device="cuda"),
                           torch.empty((b.L, len(sids), b.Hq, 128), dtype=torch.float32, device="cuda"))
        kg, vg, qg, q_rot_b, out_b = bufs[shape]
        kg.copy_(k)
        vg.copy_(v)
        qg.copy_(q)
        n0 = b.pool.launch_count()
        b.pool.step_graph(kg, vg, qg, q_rot_b, out_b)
        assert b.pool.launch_count() - n0 == a_launched
        torch.cuda.synchronize()
        a.pool.check()
        b.pool.check()
        for c in (a, b):
            for s, n in zip(sids, n_new):
                c.length[s] += n
        for l in range(a.L):
            assert torch.equal(out_a[l], out_b[l]), f"step {step} layer {l}"
    assert a.pool.seq_info(1) == b.pool.seq_info(1)
    # the graph path's last output against the fp64 oracle
    out = out_b[1].cpu().numpy()
    for i, s in enumerate(sids):
        for h in range(b.Hkv):
            qf = W.bf16_bits_to_f32(qb[1, i, h * b.hg:(h + 1) * b.hg])
            ref, _ = b.oracle_pair(s, 1, h, qf)
            assert_close_decode(out[i, h * b.hg:(h + 1) * b.hg], ref, f"seq {s} head {h}")


def test_step_graph_is_not_recorded_again_at_page_boundaries():
    """Steady decode (every sequence past the BF16 windows, one token each per step): across 130
    steps every sequence starts two new INT2 pages, which changes the INT2 unit and worker counts,
    yet the graph is recorded once; its outputs stay bit-identical to per-layer calls."""
    lengths = [700, 2047, 1350, 400]
    ids = [0, 1, 2, 3]
    a = Case(layers=2, Hq=8, Hkv=2, max_seqs=4, max_len=2400)
    b = Case(layers=2, Hq=8, Hkv=2, max_seqs=4, max_len=2400)
    for c in (a, b):
        for s in ids:
            c.add(s)
        c.step(ids, lengths)
    n_new = [1] * len(ids)
    kg = vg = qg = None
    q_rot_b = torch.empty((len(ids), b.Hq, 128), dtype=torch.float32, device="cuda")
    out_b = torch.empty((b.L, len(ids), b.Hq, 128), dtype=torch.float32, device="cuda")
    pages0 = [b.pool.seq_info(s)[2] for s in ids]
    for step in range(130):
        k, v, q, _ = _inputs(a, ids, n_new, step)
        a.pool.step_begin(ids, n_new)
        out_a = []
        for l in range(a.L):
            a.pool.append_and_demote(l, k[l], v[l])
            q_rot = a.pool.rotate_q(l, q[l])
            out_a.append(a.pool.merge(l, a.pool.decode(l, q[l], q_rot)).clone())
        b.pool.step_begin(ids, n_new)
        if kg is None:
            kg, vg, qg = torch.empty_like(k), torch.empty_like(v), torch.empty_like(q)
        kg.copy_(k)
        vg.copy_(v)
        qg.copy_(q)
        b.pool.step_graph(kg, vg, qg, q_rot_b, out_b)
        torch.cuda.synchronize()
        a.pool.check()
        b.pool.check()
        for c in (a, b):
            for s in ids:
                c.length[s] += 1
        for l in range(a.L):
            assert torch.equal(out_a[l], out_b[l]), f"step {step} layer {l}"
    assert all(b.pool.seq_info(s)[2] - p0 >= 2 for s, p0 in zip(ids, pages0))
    assert b.pool.graph_captures() == 1
