"""Torch-facing wrapper of the liboscar C ABI: allocates the device arena and step buffers with
PyTorch (device memory and streams only) and passes raw pointers to the library."""
from __future__ import annotations

import torch

from . import binding as B

HEAD_DIM = 128


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _need(t, dtype, shape, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


class Pool:
    """Mixed-precision paged KV cache for one model: BF16 sink + recent ring, rotated INT2 history."""

    def __init__(self, num_layers, num_q_heads, num_kv_heads, max_seqs, max_seq_len, max_int2_pages,
                 U_k=None, U_v=None, clip_k=None, clip_v=None, group_size=128, v_rot_absorbed=False,
                 host_only=False, lloyd_max=False, device="cuda"):
        flags = (B.OSCAR_FLAG_HOST_ONLY if host_only else 0) | (B.OSCAR_FLAG_LLOYD_MAX if lloyd_max else 0)
        self.cfg = B.OscarConfig(num_layers, num_q_heads, num_kv_heads, HEAD_DIM, 64, 64, 256, group_size,
                                 max_seqs, max_seq_len, max_int2_pages, 1 if v_rot_absorbed else 0, flags)
        self.num_layers, self.Hq, self.Hkv = num_layers, num_q_heads, num_kv_heads
        self.group_size = group_size
        self.host_only = host_only
        self.n_seqs = 0
        self.handle = None
        self._partials = None
        if host_only:
            self.arena = None
            self.handle = B.oscar_pool_create(self.cfg, None, 0, None, None, None, None, None)
            return
        shape_u = (num_layers, num_kv_heads, HEAD_DIM, HEAD_DIM)
        _need(U_k, torch.float32, shape_u, "U_k")
        _need(U_v, torch.float32, shape_u, "U_v")
        _need(clip_k, torch.float32, (num_layers, num_kv_heads), "clip_k")
        _need(clip_v, torch.float32, (num_layers, num_kv_heads), "clip_v")
        nbytes = B.oscar_arena_bytes(self.cfg)
        if nbytes == 0:
            raise B.OscarError("oscar_arena_bytes", B.OSCAR_EINVAL)
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.handle = B.oscar_pool_create(self.cfg, self.arena, nbytes, U_k, U_v, clip_k, clip_v, _stream())
        torch.cuda.current_stream().synchronize()

    # ---------------------------------------------------------------- Lloyd-Max codebook
    def set_codebook(self, a):
        """a: array-like [num_layers][num_kv_heads][2] (K, V) of interior levels (pool created with
        lloyd_max=True, before the first step)."""
        flat = [float(x) for row in a for head in row for x in head]
        B.oscar_pool_set_codebook(self.handle, flat, _stream())

    def fit_codebook(self, layer, kv_head, kv, rows, iters=50):
        """Lloyd fit of the interior level for (layer, kv_head, K|V) on bf16 rows [n][128]."""
        n = rows.shape[0]
        _need(rows, torch.bfloat16, (n, HEAD_DIM), "rows")
        scratch = torch.empty((n, HEAD_DIM), dtype=torch.float32, device=rows.device)
        return B.oscar_fit_codebook(self.handle, layer, kv_head, kv, rows, n, scratch, iters, _stream())

    # ---------------------------------------------------------------- sequences and steps
    def seq_add(self, seq_id, share_from=-1, shared_tokens=0):
        B.oscar_seq_add(self.handle, seq_id, share_from, shared_tokens)

    def seq_remove(self, seq_id):
        B.oscar_seq_remove(self.handle, seq_id)

    def seq_info(self, seq_id):
        return B.oscar_seq_info(self.handle, seq_id)

    def stats(self):
        return B.oscar_pool_get_stats(self.handle)

    def step_begin(self, seq_ids, n_new):
        B.oscar_step_begin(self.handle, seq_ids, n_new, None if self.host_only else _stream())
        self.n_seqs = len(seq_ids)
        self.total_new = int(sum(int(x) for x in n_new))

    def append_and_demote(self, layer, k_new, v_new):
        shape = (self.total_new, self.Hkv, HEAD_DIM)
        if self.total_new:
            _need(k_new, torch.bfloat16, shape, "k_new")
            _need(v_new, torch.bfloat16, shape, "v_new")
        B.oscar_append_and_demote(self.handle, layer, k_new, v_new, _stream())

    def rotate_q(self, layer, q, q_rot=None):
        _need(q, torch.bfloat16, (self.n_seqs, self.Hq, HEAD_DIM), "q")
        if q_rot is None:
            q_rot = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        _need(q_rot, torch.float32, q.shape, "q_rot")
        B.oscar_rotate_q(self.handle, layer, q, q_rot, _stream())
        return q_rot

    def partials_bytes(self):
        return B.oscar_partials_bytes(self.handle, self.n_seqs)

    def decode(self, layer, q, q_rot, partials=None):
        _need(q, torch.bfloat16, (self.n_seqs, self.Hq, HEAD_DIM), "q")
        _need(q_rot, torch.float32, (self.n_seqs, self.Hq, HEAD_DIM), "q_rot")
        nb = self.partials_bytes()
        if partials is None:
            if self._partials is None or self._partials.numel() < nb:
                self._partials = torch.empty(max(nb, 16), dtype=torch.uint8, device=q.device)
            partials = self._partials
        if partials.numel() * partials.element_size() < nb:
            raise ValueError("partials buffer too small")
        B.oscar_decode(self.handle, layer, q, q_rot, partials, _stream())
        return partials

    def merge(self, layer, partials, out=None):
        if out is None:
            out = torch.empty((self.n_seqs, self.Hq, HEAD_DIM), dtype=torch.float32, device=partials.device)
        _need(out, torch.float32, (self.n_seqs, self.Hq, HEAD_DIM), "out")
        B.oscar_merge(self.handle, layer, partials, out, _stream())
        return out

    def attend(self, layer, q):
        """rotate_q + decode + merge for one layer; returns fp32 [n_seqs, Hq, 128]."""
        q_rot = self.rotate_q(layer, q)
        part = self.decode(layer, q, q_rot)
        return self.merge(layer, part)

    def step_graph(self, k_new, v_new, q, q_rot=None, out=None):
        """Every layer's append_and_demote + rotate_q + decode + merge as one CUDA graph launch.
        k_new, v_new: bf16 [num_layers][Σn_new][Hkv][128]; q: bf16 [num_layers][n_seqs][Hq][128];
        returns out fp32 [num_layers][n_seqs][Hq][128]. Reuses the pool's graph while shapes and
        buffers stay the same (pass the same q_rot/out/partials buffers to keep them the same)."""
        NL = self.num_layers
        _need(q, torch.bfloat16, (NL, self.n_seqs, self.Hq, HEAD_DIM), "q")
        if self.total_new:
            _need(k_new, torch.bfloat16, (NL, self.total_new, self.Hkv, HEAD_DIM), "k_new")
            _need(v_new, torch.bfloat16, (NL, self.total_new, self.Hkv, HEAD_DIM), "v_new")
        if q_rot is None:
            q_rot = torch.empty(q.shape[1:], dtype=torch.float32, device=q.device)
        _need(q_rot, torch.float32, q.shape[1:], "q_rot")
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        _need(out, torch.float32, q.shape, "out")
        nb = self.partials_bytes()
        if self._partials is None or self._partials.numel() < nb:
            self._partials = torch.empty(max(nb, 16), dtype=torch.uint8, device=q.device)
        kvs = k_new[0].numel() * 2 if self.total_new else 0
        B.oscar_step_graph(self.handle, k_new if self.total_new else None, v_new if self.total_new else None, kvs,
                           q, q[0].numel() * 2, q_rot, self._partials, out, out[0].numel() * 4, _stream())
        return out

    def check(self):
        st, detail = B.oscar_check(self.handle, _stream())
        if st != B.OSCAR_OK:
            raise B.OscarError("oscar_check", st, detail)

    # ---------------------------------------------------------------- parity hooks
    def debug_rotate_rows(self, layer, kv_head, kv, x):
        n = x.shape[0]
        _need(x, torch.bfloat16, (n, HEAD_DIM), "x")
        out = torch.empty((n, HEAD_DIM), dtype=torch.float32, device=x.device)
        B.oscar_debug_rotate_rows(self.handle, layer, kv_head, kv, x, n, out, _stream())
        return out

    def debug_read_int2(self, seq_id, layer, kv_head, pos0, n):
        ng = HEAD_DIM // self.group_size
        dev = self.arena.device
        ck = torch.empty((n, 32), dtype=torch.uint8, device=dev)
        cv = torch.empty((n, 32), dtype=torch.uint8, device=dev)
        szk = torch.empty((n, ng, 2), dtype=torch.float16, device=dev)
        szv = torch.empty((n, ng, 2), dtype=torch.float16, device=dev)
        B.oscar_debug_read_int2(self.handle, seq_id, layer, kv_head, pos0, n, ck, szk, cv, szv, _stream())
        return ck, szk, cv, szv

    def debug_int2_scores(self, seq_id, layer, kv_head, q_rot_rows, pos0, n):
        """fp32 [hg][n]: q_rot_rows[h] . k_hat for INT2 tokens [pos0, pos0+n) (no 1/sqrt(d))."""
        hg = self.Hq // self.Hkv
        _need(q_rot_rows, torch.float32, (hg, HEAD_DIM), "q_rot_rows")
        out = torch.empty((hg, n), dtype=torch.float32, device=q_rot_rows.device)
        B.oscar_debug_int2_scores(self.handle, seq_id, layer, kv_head, q_rot_rows, pos0, n, out, _stream())
        return out

    def debug_read_bf16(self, seq_id, layer, kv_head, pos0, n):
        dev = self.arena.device
        k = torch.empty((n, HEAD_DIM), dtype=torch.bfloat16, device=dev)
        v = torch.empty((n, HEAD_DIM), dtype=torch.bfloat16, device=dev)
        B.oscar_debug_read_bf16(self.handle, seq_id, layer, kv_head, pos0, n, k, v, _stream())
        return k, v

    # ---------------------------------------------------------------- timing
    def timing_enable(self, kernels=True):
        """True: time every kernel kind; a list of names (binding.KERNELS) times only those; False: off."""
        if isinstance(kernels, (list, tuple)):
            mask = sum(1 << B.KERNELS.index(k) for k in kernels)
        else:
            mask = B.TIMING_ALL if kernels else 0
        B.oscar_timing_enable(self.handle, mask)

    def timing_read(self):
        return B.oscar_timing_read(self.handle)

    def launch_count(self):
        return B.oscar_launch_count(self.handle)

    def graph_captures(self):
        return B.oscar_graph_captures(self.handle)

    def int2_workers(self):
        """INT2 decode workers (split-K segments) of the current step."""
        return B.oscar_step_int2_workers(self.handle)

    def close(self):
        if self.handle is not None:
            B.oscar_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
