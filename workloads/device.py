"""Device twin of the synthetic generator (workloads/synth.cu), built in-tree with nvcc and
called through ctypes. Input generation only."""
from __future__ import annotations

import ctypes
import os
import platform
import shutil
import subprocess

import numpy as np

from .synth import INV_SIGMA_F32, OUTLIER_SCALE_F32, TAG_KV

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "synth.cu")
LIB = os.path.join(HERE, "_lib", "libsynth.so")
_lib = None


def build_synth(force: bool = False) -> str:
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    stamp = LIB + ".machine"
    if (not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.exists(stamp) and open(stamp).read().strip() == platform.machine()):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "shared", "-Xlinker", "-rpath," + os.path.join(home, "lib64"), SRC, "-o", LIB + ".tmp"]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("libsynth build failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(LIB + ".tmp", LIB)
    with open(stamp, "w") as f:
        f.write(platform.machine())
    return LIB


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("libsynth.so is not built (call workloads.device.build_synth())")
        L = ctypes.CDLL(LIB)
        L.synth_kv_bf16.restype = ctypes.c_int
        L.synth_kv_bf16.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_void_p]
        L.read_stream.restype = ctypes.c_int
        L.read_stream.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
        _lib = L
    return _lib


def read_stream_gbs(dev, gib=8, reps=5):
    """Read-only HBM bandwidth: best of `reps` timed passes (CUDA events) of a streaming-read kernel
    over a `gib` GiB buffer (far larger than L2), after one untimed pass. Returns GB/s."""
    import torch

    nbytes = gib << 30
    buf = torch.ones(nbytes // 2, dtype=torch.int16, device=dev)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks = 4 * n_sm
    out = torch.empty(blocks * 512, dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream(dev)
    best = None
    for r in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        rc = lib().read_stream(ctypes.c_void_p(buf.data_ptr()), ctypes.c_ulonglong(nbytes),
                               ctypes.c_void_p(out.data_ptr()), blocks, ctypes.c_void_p(st.cuda_stream))
        e1.record(st)
        if rc != 0:
            raise RuntimeError(f"read_stream failed with CUDA error {rc}")
        e1.synchronize()
        if r:
            gbs = nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9
            best = gbs if best is None else max(best, gbs)
    del buf, out
    torch.cuda.empty_cache()
    return best


def fill_kv(out, seed, seq_key, layer, kv, head0, n_heads, pos0, n_pos, mask_dev, stream):
    """Write bf16 rows [n_pos][n_heads][128] of K (kv=0) or V (kv=1) into the device buffer
    ``out`` (a torch CUDA tensor), identical to workloads.synth.kv_rows_bf16."""
    rc = lib().synth_kv_bf16(ctypes.c_void_p(out.data_ptr()), ctypes.c_ulonglong(seed), TAG_KV, seq_key,
                             layer, kv, head0, n_heads, pos0, n_pos,
                             ctypes.c_void_p(mask_dev.data_ptr() if mask_dev is not None else 0),
                             ctypes.c_float(float(INV_SIGMA_F32)), ctypes.c_float(float(OUTLIER_SCALE_F32)),
                             ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_kv_bf16 failed with CUDA error {rc}")
