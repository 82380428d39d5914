"""Pipe-rate probes (libdwprobe.so, built from peak_probes.cu; not part of the
convolution library).

fma_rates()       FP32 FFMA, packed FFMA2 and mixed-precision f16 / bf16 FMA
                  rates in TFLOP/s: the measured counterparts of the derived
                  FP32 FMA peak that the CUDA-core kernels' roofline uses.
mma_sync_rate()   warp-level mma.sync m16n8k16 bf16 rate.
tcgen05_rates()   tcgen05.mma kind::f16 rates over the M x N shapes the
                  Toeplitz packing could use.

    python -m depthwise_convolution_gb300.probes [fma|mma|tcgen05|all]

prints one JSON object.
"""
from __future__ import annotations

import ctypes
import json
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "peak_probes.cu")
LIB = os.path.join(HERE, "_build", "libdwprobe.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile libdwprobe.so for sm_103a if the source is newer (nvcc)."""
    from .. import build as lib_build
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [lib_build.nvcc()] + lib_build.ARCH + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                                                  SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on peak_probes.cu:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        D, I, U = ctypes.POINTER(ctypes.c_double), ctypes.c_int, ctypes.POINTER(ctypes.c_uint)
        lib.dwp_fma_rate.argtypes = [I, I, I, D]
        lib.dwp_mma_sync_rate.argtypes = [I, I, D]
        lib.dwp_tcgen05_rate.argtypes = [I, I, I, I, I, I, D, U]
        for f in (lib.dwp_fma_rate, lib.dwp_mma_sync_rate, lib.dwp_tcgen05_rate):
            f.restype = I
        _lib = lib
    return _lib


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what}: probe failed (code {rc})")


FMA_KINDS = {"ffma_f32": 0, "ffma2_f32x2": 1, "fma_f32_f16": 2, "fma_f32_bf16": 3}


def fma_rates(warps=(8, 16, 32), iters=4096) -> dict:
    """Best TFLOP/s of each FMA form over a few warps-per-SM counts."""
    lib = _load()
    out = {}
    for name, kind in FMA_KINDS.items():
        best = 0.0
        for w in warps:
            v = ctypes.c_double()
            _check(lib.dwp_fma_rate(kind, w, iters, ctypes.byref(v)), name)
            best = max(best, v.value)
        out[name] = round(best, 2)
    return out


def mma_sync_rate(warps=(4, 8, 16), iters=2048) -> dict:
    lib = _load()
    out = {}
    for w in warps:
        v = ctypes.c_double()
        _check(lib.dwp_mma_sync_rate(w, iters, ctypes.byref(v)), "mma.sync")
        out[f"warps_per_sm_{w}"] = round(v.value, 1)
    return out


# (M, N, MMAs per commit, accumulators per warp, issuing warps)
TCGEN05_SHAPES = [(128, 256, 8, 1, 1), (128, 128, 16, 2, 1), (128, 64, 32, 1, 4), (128, 32, 32, 2, 4),
                  (128, 16, 32, 4, 4), (64, 64, 32, 1, 4), (64, 16, 32, 4, 4), (64, 8, 32, 8, 4), (64, 8, 32, 1, 1)]


def tcgen05_rates(iters=200) -> dict:
    lib = _load()
    out = {}
    for (M, N, per, nd, nw) in TCGEN05_SHAPES:
        v, to = ctypes.c_double(), ctypes.c_uint()
        _check(lib.dwp_tcgen05_rate(M, N, per, nd, nw, iters, ctypes.byref(v), ctypes.byref(to)), "tcgen05")
        out[f"M{M}_N{N}_warps{nw}"] = None if to.value else round(v.value, 1)
    return out


def main(argv):
    what = argv[1] if len(argv) > 1 else "all"
    res = {}
    if what in ("fma", "all"):
        res["fma_tflops"] = fma_rates()
    if what in ("mma", "all"):
        res["mma_sync_tflops"] = mma_sync_rate()
    if what in ("tcgen05", "all"):
        res["tcgen05_tflops"] = tcgen05_rates()
    print(json.dumps(res))


if __name__ == "__main__":
    main(sys.argv)
