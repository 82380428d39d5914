"""Seeded synthetic inputs for the depthwise-convolution workloads.

This module only draws random numbers and casts them to the storage dtype; it
holds none of the convolution's arithmetic.  Tests, the benchmark and the
oracle all consume what it returns, so both sides of every parity check see
the same quantised values.

Recipe (per tensor): numpy PCG64 seeded with (workload seed, tensor id), drawn
as float32 N(0, sigma^2) or as uniform integers over an inclusive range, then
cast once to the workload's dtype (round-to-nearest-even for 16-bit floats
and for FP8 E4M3, whose inputs stay far below its largest value, 448).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

_TORCH_DTYPES = {
    "int8": torch.int8,
    "fp32": torch.float32,
    "fp16": torch.float16,
    "bf16": torch.bfloat16,
    "fp8": getattr(torch, "float8_e4m3fn", None),  # E4M3 inputs of the forward pass
}

# Tensor ids within a workload's seed sequence.
_X, _W, _B, _DY = 0, 1, 2, 3
_PRE, _POST = 4, 6  # scale at the id, shift at id + 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "int8" | "fp32" | "fp16" | "bf16"
    N: int
    H: int
    W: int
    C: int
    FH: int
    FW: int
    stride: int
    dilation: int
    pad: int
    bias: bool                 # forward adds a bias
    passes: tuple              # subset of ("fwd", "dgrad", "wgrad")
    seed: int
    x_sigma: float = 1.0
    dy_sigma: float = 1.0
    bias_sigma: float = math.sqrt(0.1)

    @property
    def w_sigma(self) -> float:
        # N(0, 1/(FH*FW)): variance 1/(FH*FW), the fan-in scaling of the filter.
        return 1.0 / math.sqrt(self.FH * self.FW)

    def with_batch(self, N: int) -> "Workload":
        return dataclasses.replace(self, N=N, name=f"{self.name}[N={N}]")

    def shape_args(self):
        return (self.N, self.H, self.W, self.C, self.FH, self.FW,
                self.stride, self.dilation, self.pad)


def _rng(seed: int, tensor: int, part: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, tensor, part])


def normal(shape, sigma: float, seed: int, tensor: int) -> np.ndarray:
    """float32 N(0, sigma^2) draws, generated in chunks along the first axis."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.float32)
    if out.size == 0:
        return out
    rows = shape[0]
    per_row = out.size // rows
    chunk = max(1, (1 << 24) // max(1, per_row))
    flat = out.reshape(rows, per_row)
    for part, r0 in enumerate(range(0, rows, chunk)):
        r1 = min(rows, r0 + chunk)
        g = _rng(seed, tensor, part)
        flat[r0:r1] = g.standard_normal((r1 - r0, per_row), dtype=np.float32)
    if sigma != 1.0:
        out *= np.float32(sigma)
    return out


def uniform_int(shape, lo: int, hi: int, seed: int, tensor: int) -> np.ndarray:
    """Uniform integers over the inclusive range [lo, hi]."""
    return _rng(seed, tensor).integers(lo, hi, size=shape, endpoint=True, dtype=np.int64)


def _cast(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(a).to(_TORCH_DTYPES[dtype])


def make_inputs(wl: Workload, dy_hw=None) -> dict:
    """CPU tensors in storage dtype: x, w, bias (or None), dy (if a backward pass).

    ``dy_hw`` = (OH, OW), the spatial size of the forward output, which the
    caller computes; it is required when the workload has a backward pass.

    int8 workloads: x, w int8 uniform over [-128, 127], bias int32 uniform over
    [-1000, 1000].  Floating workloads: x ~ N(0, x_sigma^2), w ~ N(0, 1/(FH FW)),
    dy ~ N(0, dy_sigma^2) in the workload dtype; bias fp32 ~ N(0, 0.1).
    """
    out = {}
    if wl.dtype == "int8":
        out["x"] = torch.from_numpy(uniform_int((wl.N, wl.H, wl.W, wl.C), -128, 127, wl.seed, _X)).to(torch.int8)
        out["w"] = torch.from_numpy(uniform_int((wl.FH, wl.FW, wl.C), -128, 127, wl.seed, _W)).to(torch.int8)
        out["bias"] = (torch.from_numpy(uniform_int((wl.C,), -1000, 1000, wl.seed, _B)).to(torch.int32)
                       if wl.bias else None)
        out["dy"] = None
        return out
    out["x"] = _cast(normal((wl.N, wl.H, wl.W, wl.C), wl.x_sigma, wl.seed, _X), wl.dtype)
    out["w"] = _cast(normal((wl.FH, wl.FW, wl.C), wl.w_sigma, wl.seed, _W), wl.dtype)
    out["bias"] = (torch.from_numpy(normal((wl.C,), wl.bias_sigma, wl.seed, _B)) if wl.bias else None)
    needs_dy = any(p in wl.passes for p in ("dgrad", "wgrad"))
    if needs_dy and dy_hw is None:
        raise ValueError("dy_hw=(OH, OW) is required for a workload with a backward pass")
    out["dy"] = (_cast(normal((wl.N, dy_hw[0], dy_hw[1], wl.C), wl.dy_sigma, wl.seed, _DY), wl.dtype)
                 if needs_dy else None)
    return out


def make_affine(C: int, seed: int, stage: str) -> tuple:
    """Per-channel (scale, shift) float32 CPU vectors for a fused forward pass,
    stage "pre" (the BN before the convolution) or "post" (after it): scale
    ~ N(1, 0.5^2) (a folded BN's gamma / sqrt(var + eps), sign changes
    included), shift ~ N(0, 0.5^2)."""
    base = {"pre": _PRE, "post": _POST}[stage]
    scale = normal((C,), 0.5, seed, base) + np.float32(1.0)
    shift = normal((C,), 0.5, seed, base + 1)
    return torch.from_numpy(scale.astype(np.float32)), torch.from_numpy(shift.astype(np.float32))


# The five workloads: shapes, distributions and seeds.
WORKLOADS = {
    "int8-fwd-3x3-1x8x8x5": Workload(
        "int8-fwd-3x3-1x8x8x5", "int8", 1, 8, 8, 5, 3, 3, 1, 1, 1, True, ("fwd",), 1),
    "fp32-fwd-7x7-64x56x56x128": Workload(
        "fp32-fwd-7x7-64x56x56x128", "fp32", 64, 56, 56, 128, 7, 7, 1, 1, 3, True, ("fwd",), 2),
    "bf16-fwd-31x31-32x56x56x128": Workload(
        "bf16-fwd-31x31-32x56x56x128", "bf16", 32, 56, 56, 128, 31, 31, 1, 1, 15, True, ("fwd",), 3),
    "fp16-train-7x7-128x56x56x96": Workload(
        "fp16-train-7x7-128x56x56x96", "fp16", 128, 56, 56, 96, 7, 7, 1, 1, 3, False,
        ("fwd", "dgrad", "wgrad"), 4),
}

# bf16 stage sweep: four 7x7 stages and one 5x5 stride-2 dilation-2 layer.
STAGE_SWEEP = [
    Workload("bf16-train-7x7-128x56x56x96", "bf16", 128, 56, 56, 96, 7, 7, 1, 1, 3, False,
             ("fwd", "dgrad", "wgrad"), 51),
    Workload("bf16-train-7x7-128x28x28x192", "bf16", 128, 28, 28, 192, 7, 7, 1, 1, 3, False,
             ("fwd", "dgrad", "wgrad"), 52),
    Workload("bf16-train-7x7-128x14x14x384", "bf16", 128, 14, 14, 384, 7, 7, 1, 1, 3, False,
             ("fwd", "dgrad", "wgrad"), 53),
    Workload("bf16-train-7x7-128x7x7x768", "bf16", 128, 7, 7, 768, 7, 7, 1, 1, 3, False,
             ("fwd", "dgrad", "wgrad"), 54),
    Workload("bf16-train-5x5s2d2-64x112x112x64", "bf16", 64, 112, 112, 64, 5, 5, 2, 2, 4, False,
             ("fwd", "dgrad", "wgrad"), 55),
]
for _wl in STAGE_SWEEP:
    WORKLOADS[_wl.name] = _wl

# Further layers bench.py times next to the workloads (not configurations of
# the benchmark): the stride-2 down-sampling layer, and odd square filters of
# the Flash-DWC §6.1 sweep (3 to 51) on the 31x31 layer's shape.
EXTRA_LAYERS = {
    "bf16-train-3x3s2-128x56x56x96": Workload(
        "bf16-train-3x3s2-128x56x56x96", "bf16", 128, 56, 56, 96, 3, 3, 2, 1, 1, False,
        ("fwd", "dgrad", "wgrad"), 61),
}
for _i, _F in enumerate((9, 15, 21, 27)):
    _name = f"bf16-fwd-{_F}x{_F}-32x56x56x128"
    EXTRA_LAYERS[_name] = Workload(_name, "bf16", 32, 56, 56, 128, _F, _F, 1, 1, _F // 2, True, ("fwd",), 62 + _i)
