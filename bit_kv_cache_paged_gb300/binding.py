"""ctypes binding of liboscar's C ABI (include/oscar.h): the same names, argument marshalling
only. Every step of the decode path runs in liboscar's CUDA kernels; there is no Python or CPU
fallback, and loading fails loudly when the library is missing."""
from __future__ import annotations

import ctypes
import os
import re

from .build import LIB, ROOT

c_i32, c_i64, c_sz, c_vp, c_u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_uint32

STATUS = {0: "OSCAR_OK", 1: "OSCAR_EINVAL", 2: "OSCAR_ENOMEM", 3: "OSCAR_EFULL", 4: "OSCAR_ECUDA",
          5: "OSCAR_EDEVICE", 6: "OSCAR_ETIMEOUT", 7: "OSCAR_ESTATE"}
OSCAR_OK, OSCAR_EINVAL, OSCAR_ENOMEM, OSCAR_EFULL, OSCAR_ECUDA, OSCAR_EDEVICE, OSCAR_ETIMEOUT, OSCAR_ESTATE = range(8)
OSCAR_FLAG_HOST_ONLY = 1
OSCAR_FLAG_LLOYD_MAX = 2
DEVERR_PAGE, DEVERR_SCALE, DEVERR_TIMEOUT, DEVERR_INPUT = 1, 2, 4, 8
NOALLOC_PARTIALS_MAX_BYTES = 16 << 20  # OSCAR_NOALLOC_PARTIALS_MAX_BYTES
KERNELS = ["demote", "append", "rotate_q", "decode_int2", "decode_bf16", "merge"]


class OscarError(RuntimeError):
    def __init__(self, fn, status, detail=0):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}" + (f" (device error bits 0x{detail:x})" if detail else ""))
        self.status = status
        self.detail = detail


class OscarConfig(ctypes.Structure):
    _fields_ = [("num_layers", c_i32), ("num_q_heads", c_i32), ("num_kv_heads", c_i32), ("head_dim", c_i32),
                ("page_size", c_i32), ("sink_size", c_i32), ("recent_size", c_i32), ("group_size", c_i32),
                ("max_seqs", c_i32), ("max_seq_len", c_i32), ("max_int2_pages", c_i64),
                ("v_rot_absorbed", c_i32), ("flags", c_i32)]


class OscarPoolStats(ctypes.Structure):
    _fields_ = [("int2_pages_used", c_i64), ("int2_pages_free", c_i64), ("sink_pages_used", c_i32),
                ("seqs_active", c_i32), ("bf16_bytes_per_token", c_i64), ("int2_bytes_per_token", c_i64)]


_SIGS = {
    "oscar_version": (ctypes.c_char_p, []),
    "oscar_arena_bytes": (c_sz, [ctypes.POINTER(OscarConfig)]),
    "oscar_pool_create": (c_i32, [ctypes.POINTER(OscarConfig), c_vp, c_sz, c_vp, c_vp, c_vp, c_vp, c_vp,
                                  ctypes.POINTER(c_vp)]),
    "oscar_pool_destroy": (c_i32, [c_vp]),
    "oscar_pool_set_codebook": (c_i32, [c_vp, ctypes.POINTER(ctypes.c_float), c_vp]),
    "oscar_fit_codebook": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_vp, c_i32, c_vp, c_i32,
                                   ctypes.POINTER(ctypes.c_float), c_vp]),
    "oscar_seq_add": (c_i32, [c_vp, c_i32, c_i32, c_i32]),
    "oscar_seq_remove": (c_i32, [c_vp, c_i32]),
    "oscar_step_begin": (c_i32, [c_vp, ctypes.POINTER(c_i32), ctypes.POINTER(c_i32), c_i32, c_vp]),
    "oscar_append_and_demote": (c_i32, [c_vp, c_i32, c_vp, c_vp, c_vp]),
    "oscar_rotate_q": (c_i32, [c_vp, c_i32, c_vp, c_vp, c_vp]),
    "oscar_decode": (c_i32, [c_vp, c_i32, c_vp, c_vp, c_vp, c_vp]),
    "oscar_merge": (c_i32, [c_vp, c_i32, c_vp, c_vp, c_vp]),
    "oscar_partials_bytes": (c_sz, [c_vp, c_i32]),
    "oscar_bf16_partials_bytes": (c_sz, [c_i32, c_i32, c_i32, c_i32]),
    "oscar_bf16_pack": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_vp, c_i64, c_vp, c_vp, c_vp]),
    "oscar_bf16_decode": (c_i32, [c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_i64, c_vp, c_i32, c_vp, c_vp, c_vp,
                                  c_sz, c_vp, c_vp, c_vp]),
    "oscar_step_graph": (c_i32, [c_vp, c_vp, c_vp, c_sz, c_vp, c_sz, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "oscar_decode_merge_noalloc": (c_i32, [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp]),
    "oscar_check": (c_i32, [c_vp, c_vp, ctypes.POINTER(c_u32)]),
    "oscar_seq_info": (c_i32, [c_vp, c_i32, ctypes.POINTER(c_i32), ctypes.POINTER(c_i32), ctypes.POINTER(c_i32)]),
    "oscar_pool_get_stats": (c_i32, [c_vp, ctypes.POINTER(OscarPoolStats)]),
    "oscar_debug_rotate_rows": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp]),
    "oscar_debug_read_int2": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "oscar_debug_read_bf16": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "oscar_debug_timeout_selftest": (c_i32, [c_vp, c_vp]),
    "oscar_debug_set_page_entry": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_vp]),
    "oscar_debug_restore_page_table": (c_i32, [c_vp, c_i32, c_vp]),
    "oscar_debug_int2_scores": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_vp, c_i32, c_i32, c_vp, c_vp]),
    "oscar_timing_enable": (c_i32, [c_vp, c_i32]),
    "oscar_timing_read": (c_i32, [c_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_i64)]),
    "oscar_launch_count": (c_i64, [c_vp]),
    "oscar_graph_captures": (c_i64, [c_vp]),
    "oscar_step_int2_workers": (c_i32, [c_vp]),
}

_lib = None


def header_symbols():
    """Names of the functions include/oscar.h declares."""
    text = open(os.path.join(ROOT, "include", "oscar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oscar_[a-z0-9_]+)\s*\(", text)))


def lib():
    """Load liboscar.so (built in-tree). Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"liboscar is not built ({LIB} missing); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _check(fn, st):
    if st != OSCAR_OK:
        raise OscarError(fn, st)


def oscar_version():
    return lib().oscar_version().decode()


def oscar_arena_bytes(cfg: OscarConfig) -> int:
    return lib().oscar_arena_bytes(ctypes.byref(cfg))


def oscar_pool_create(cfg, arena, arena_bytes, U_k, U_v, clip_k, clip_v, stream):
    out = c_vp()
    _check("oscar_pool_create", lib().oscar_pool_create(ctypes.byref(cfg), _ptr(arena), arena_bytes, _ptr(U_k),
                                                        _ptr(U_v), _ptr(clip_k), _ptr(clip_v), stream,
                                                        ctypes.byref(out)))
    return out.value


def oscar_pool_destroy(pool):
    _check("oscar_pool_destroy", lib().oscar_pool_destroy(pool))


def oscar_pool_set_codebook(pool, a_values, stream):
    """a_values: flat host sequence of num_layers * num_kv_heads * 2 floats (K then V per head)."""
    vals = [float(x) for x in a_values]
    arr = (ctypes.c_float * len(vals))(*vals)
    _check("oscar_pool_set_codebook", lib().oscar_pool_set_codebook(pool, arr, stream))


def oscar_fit_codebook(pool, layer, kv_head, kv, rows, n, scratch, iters, stream) -> float:
    a = ctypes.c_float(0.0)
    _check("oscar_fit_codebook", lib().oscar_fit_codebook(pool, layer, kv_head, kv, _ptr(rows), n, _ptr(scratch),
                                                          iters, ctypes.byref(a), stream))
    return a.value


def oscar_seq_add(pool, seq_id, share_from=-1, shared_tokens=0):
    _check("oscar_seq_add", lib().oscar_seq_add(pool, seq_id, share_from, shared_tokens))


def oscar_seq_remove(pool, seq_id):
    _check("oscar_seq_remove", lib().oscar_seq_remove(pool, seq_id))


def oscar_step_begin(pool, seq_ids, n_new, stream):
    n = len(seq_ids)
    a = (c_i32 * n)(*[int(x) for x in seq_ids])
    b = (c_i32 * n)(*[int(x) for x in n_new])
    _check("oscar_step_begin", lib().oscar_step_begin(pool, a, b, n, stream))


def oscar_append_and_demote(pool, layer, k_new, v_new, stream):
    _check("oscar_append_and_demote", lib().oscar_append_and_demote(pool, layer, _ptr(k_new), _ptr(v_new), stream))


def oscar_rotate_q(pool, layer, q, q_rot, stream):
    _check("oscar_rotate_q", lib().oscar_rotate_q(pool, layer, _ptr(q), _ptr(q_rot), stream))


def oscar_decode(pool, layer, q, q_rot, partials, stream):
    _check("oscar_decode", lib().oscar_decode(pool, layer, _ptr(q), _ptr(q_rot), _ptr(partials), stream))


def oscar_merge(pool, layer, partials, out, stream):
    _check("oscar_merge", lib().oscar_merge(pool, layer, _ptr(partials), _ptr(out), stream))


def oscar_step_graph(pool, k_new, v_new, kv_layer_stride, q, q_layer_stride, q_rot, partials, out,
                     out_layer_stride, stream):
    _check("oscar_step_graph", lib().oscar_step_graph(pool, _ptr(k_new), _ptr(v_new), kv_layer_stride, _ptr(q),
                                                      q_layer_stride, _ptr(q_rot), _ptr(partials), _ptr(out),
                                                      out_layer_stride, stream))


def oscar_bf16_partials_bytes(num_q_heads, num_kv_heads, n_seqs, max_len) -> int:
    return lib().oscar_bf16_partials_bytes(num_q_heads, num_kv_heads, n_seqs, max_len)


def oscar_bf16_pack(rows, n, pos0, num_kv_heads, page_table_row, n_pages_total, pages, err, stream):
    _check("oscar_bf16_pack", lib().oscar_bf16_pack(_ptr(rows), n, pos0, num_kv_heads, _ptr(page_table_row),
                                                    n_pages_total, _ptr(pages), _ptr(err), stream))


def oscar_bf16_decode(num_q_heads, num_kv_heads, n_seqs, max_len, k_pages, v_pages, n_pages_total, page_table,
                      max_pages_per_seq, lengths, q, partials, partials_bytes, out, err, stream):
    _check("oscar_bf16_decode", lib().oscar_bf16_decode(num_q_heads, num_kv_heads, n_seqs, max_len, _ptr(k_pages),
                                                        _ptr(v_pages), n_pages_total, _ptr(page_table),
                                                        max_pages_per_seq, _ptr(lengths), _ptr(q), _ptr(partials),
                                                        partials_bytes, _ptr(out), _ptr(err), stream))


def oscar_partials_bytes(pool, n_seqs) -> int:
    return lib().oscar_partials_bytes(pool, n_seqs)


def oscar_decode_merge_noalloc(pool, layer, n_seqs, q, q_rot, out, stream):
    """oscar_decode + oscar_merge with the partials in liboscar's own device array (no allocation;
    calls overlapping on one device race on that array)."""
    _check("oscar_decode_merge_noalloc", lib().oscar_decode_merge_noalloc(pool, layer, n_seqs, _ptr(q), _ptr(q_rot),
                                                                          _ptr(out), stream))


def oscar_check(pool, stream):
    """Returns (status, detail bits) without raising."""
    d = c_u32(0)
    st = lib().oscar_check(pool, stream, ctypes.byref(d))
    return st, d.value


def oscar_seq_info(pool, seq_id):
    L, F, n = c_i32(), c_i32(), c_i32()
    _check("oscar_seq_info", lib().oscar_seq_info(pool, seq_id, ctypes.byref(L), ctypes.byref(F), ctypes.byref(n)))
    return L.value, F.value, n.value


def oscar_pool_get_stats(pool) -> dict:
    s = OscarPoolStats()
    _check("oscar_pool_get_stats", lib().oscar_pool_get_stats(pool, ctypes.byref(s)))
    return {k: getattr(s, k) for k, _ in OscarPoolStats._fields_}


def oscar_debug_rotate_rows(pool, layer, kv_head, kv, x, n, out, stream):
    _check("oscar_debug_rotate_rows", lib().oscar_debug_rotate_rows(pool, layer, kv_head, kv, _ptr(x), n, _ptr(out), stream))


def oscar_debug_read_int2(pool, seq_id, layer, kv_head, pos0, n, codes_k, sz_k, codes_v, sz_v, stream):
    _check("oscar_debug_read_int2", lib().oscar_debug_read_int2(pool, seq_id, layer, kv_head, pos0, n, _ptr(codes_k),
                                                                _ptr(sz_k), _ptr(codes_v), _ptr(sz_v), stream))


def oscar_debug_read_bf16(pool, seq_id, layer, kv_head, pos0, n, k_out, v_out, stream):
    _check("oscar_debug_read_bf16", lib().oscar_debug_read_bf16(pool, seq_id, layer, kv_head, pos0, n, _ptr(k_out),
                                                                _ptr(v_out), stream))


def oscar_debug_int2_scores(pool, seq_id, layer, kv_head, q_rot, pos0, n, out, stream):
    _check("oscar_debug_int2_scores", lib().oscar_debug_int2_scores(pool, seq_id, layer, kv_head, _ptr(q_rot), pos0,
                                                                    n, _ptr(out), stream))


def oscar_debug_timeout_selftest(pool, stream):
    _check("oscar_debug_timeout_selftest", lib().oscar_debug_timeout_selftest(pool, stream))


def oscar_debug_set_page_entry(pool, seq_id, page, value, stream):
    _check("oscar_debug_set_page_entry", lib().oscar_debug_set_page_entry(pool, seq_id, page, value, stream))


def oscar_debug_restore_page_table(pool, seq_id, stream):
    _check("oscar_debug_restore_page_table", lib().oscar_debug_restore_page_table(pool, seq_id, stream))


TIMING_ALL = (1 << len(KERNELS)) - 1


def oscar_timing_enable(pool, kernel_mask):
    """kernel_mask: bit k times kernel kind KERNELS[k]; True = all kinds, False/0 = off."""
    if kernel_mask is True:
        kernel_mask = TIMING_ALL
    _check("oscar_timing_enable", lib().oscar_timing_enable(pool, int(kernel_mask)))


def oscar_timing_read(pool):
    ms = (ctypes.c_double * len(KERNELS))()
    n = (c_i64 * len(KERNELS))()
    _check("oscar_timing_read", lib().oscar_timing_read(pool, ms, n))
    return {k: (ms[i], n[i]) for i, k in enumerate(KERNELS)}


def oscar_launch_count(pool) -> int:
    return lib().oscar_launch_count(pool)


def oscar_graph_captures(pool) -> int:
    return lib().oscar_graph_captures(pool)


def oscar_step_int2_workers(pool) -> int:
    return lib().oscar_step_int2_workers(pool)
