"""Build liboscar.so (sm_103a) in-tree with nvcc: one translation unit per source file,
compiled in parallel, linked against the shared CUDA runtime (the one PyTorch also loads)."""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build", platform.machine(), "oscar")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "liboscar.so")
SOURCES = ["pool.cpp", "demote.cu", "decode_int2.cu", "decode_bf16_merge.cu", "decode_noalloc.cu", "bf16_baseline.cu", "demote_tc.cu"]
HEADERS = ["oscar_internal.h", "device_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: liboscar needs the CUDA toolkit to build")


def cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


STAMP = LIB + ".machine"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    if target == LIB and (not os.path.exists(STAMP) or open(STAMP).read().strip() != platform.machine()):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False) -> str:
    nvcc = nvcc_path()
    home = cuda_home(nvcc)
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "oscar.h")]
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3,-ffp-contract=off",
                     "-I" + os.path.join(ROOT, "include")]
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    objs, procs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            cmd = [nvcc] + common + ["-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose or ptxas_info:
            sys.stdout.write(text)
    if failed:
        raise RuntimeError("liboscar build failed:\n" + "\n".join(f"--- {s}\n{t}" for s, t in failed))
    if force or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
            "-Xlinker", "-rpath," + os.path.join(home, "lib64")]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("liboscar link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, LIB)
        with open(STAMP, "w") as f:
            f.write(platform.machine())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, ptxas_info="--ptxas" in sys.argv))
