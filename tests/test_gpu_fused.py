"""Fused forward pass (BN+Act prologue, affine+activation epilogue; Flash-DWC
§5.2 "Kernel fusion") against oracle.fwd_fused, element by element, on every
kernel family that provides it, and on the direct kernel that takes the
shapes the others decline.
"""
from __future__ import annotations

import pytest
import torch

from depthwise_convolution_gb300 import synthetic as syn
from parity import check_fused, random_inputs

pytestmark = pytest.mark.gpu

# (dtype, (N, H, W, C, FH, FW, S, D, P), kernel family expected with a prologue)
CASES = [
    ("bf16", (2, 19, 45, 40, 7, 7, 1, 1, 3), "tiled_mma"),     # G = 8, channel tail, ragged rows
    ("fp16", (2, 22, 20, 32, 5, 5, 1, 1, 2), "tiled_mma"),     # G = 4
    ("bf16", (3, 9, 12, 48, 3, 3, 1, 1, 1), "tiled_mma"),      # G = 2, two images per unit, odd N
    ("fp16", (2, 18, 24, 16, 31, 31, 1, 1, 15), "tiled_mma_large"),
    ("bf16", (2, 20, 40, 8, 13, 13, 1, 1, 6), "tiled_mma_large"),
    ("bf16", (4, 7, 7, 64, 7, 7, 1, 1, 3), "smallmap"),        # 7x7 maps, "same": whole-map kernel
    ("fp16", (5, 7, 7, 40, 5, 5, 1, 1, 2), "smallmap"),        # 5 images (slots of 4), 20 channel pairs
    ("fp32", (3, 7, 7, 96, 3, 3, 1, 1, 1), "smallmap"),        # fp32: one channel per lane
    ("bf16", (2, 7, 7, 32, 7, 7, 1, 1, 2), "tiled_small"),     # 7x7 maps, other padding: CUDA-core kernel
    ("fp32", (2, 17, 23, 36, 7, 7, 1, 1, 3), "tiled_small"),
    ("fp32", (2, 12, 15, 32, 3, 5, 1, 1, (1, 2)), "tiled_small"),
    ("fp16", (2, 24, 24, 32, 3, 3, 2, 2, 2), "tiled_mma"),     # stride 2 dilation 2: even sub-grid
    ("fp32", (2, 13, 13, 12, 3, 3, 2, 1, 1), "strided_fwd"),   # stride 2: the strided kernel
    ("bf16", (3, 29, 30, 64, 7, 7, 2, 1, 3), "strided_fwd"),   # stride 2, 7x7, ragged tiles
    ("fp16", (2, 16, 21, 32, 5, 5, 2, 1, (2, 1)), "strided_fwd"),  # stride 2, unequal padding
    ("bf16", (1, 9, 11, 5, 3, 3, 1, 1, 1), "direct_fwd"),      # odd C: direct kernel
    ("fp32", (1, 20, 24, 32, 9, 9, 1, 1, 4), "direct_fwd"),    # large filter + prologue: direct
]
# epilogue-only families where they differ from the prologue ones
POST_ONLY = {("fp32", (1, 20, 24, 32, 9, 9, 1, 1, 4)): "tiled_large"}

ACTS = ["relu", "relu6", "silu", "gelu"]


def _ids(c):
    dt, (N, H, W, C, FH, FW, S, D, P), fam = c
    return f"{dt}-{N}x{H}x{W}x{C}-{FH}x{FW}-s{S}d{D}p{P}-{fam}"


def _affine(C, seed, stage, act, scale=True, shift=True):
    s, t = syn.make_affine(C, seed, stage)
    return (s if scale else None, t if shift else None, act)


@pytest.mark.parametrize("case", CASES, ids=_ids)
@pytest.mark.parametrize("mode", ["pre", "post", "both"])
def test_fused_matches_oracle(case, mode):
    dt, shape, fam = case
    N, H, W, C, FH, FW, S, D, P = shape
    d = random_inputs(dt, N, H, W, C, FH, FW, S, D, P, seed=31)
    k = sum(shape[:6]) % len(ACTS)
    pre = _affine(C, 5, "pre", ACTS[k]) if mode in ("pre", "both") else None
    post = _affine(C, 6, "post", ACTS[(k + 1) % len(ACTS)]) if mode in ("post", "both") else None
    kernel = check_fused(d, dt, S, D, P, pre=pre, post=post, what=f"fused-{mode}")
    expect = POST_ONLY.get((dt, shape), fam) if mode == "post" else fam
    assert kernel == expect


@pytest.mark.parametrize("act", ["none"] + ACTS)
@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32"])
def test_every_activation_both_sides(dt, act):
    shape = (2, 14, 34, 32, 7, 7, 1, 1, 3)
    d = random_inputs(dt, *shape, seed=41)
    C = shape[3]
    check_fused(d, dt, 1, 1, 3, pre=_affine(C, 7, "pre", act), post=_affine(C, 8, "post", act),
                what=f"act-{act}")


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_partial_affine_and_identity(dt):
    """Scale only, shift only, and the all-default call (a plain forward pass)."""
    shape = (2, 12, 40, 32, 5, 5, 1, 1, 2)
    d = random_inputs(dt, *shape, seed=43)
    C = shape[3]
    check_fused(d, dt, 1, 1, 2, pre=_affine(C, 9, "pre", "none", shift=False),
                post=_affine(C, 10, "post", "relu", scale=False), what="partial")
    check_fused(d, dt, 1, 1, 2, pre=_affine(C, 11, "pre", "relu6", scale=False),
                post=_affine(C, 12, "post", "none", shift=False), what="partial2")
    from depthwise_convolution_gb300 import ops
    x, w, b = d["x"].cuda(), d["w"].cuda(), d["bias"].cuda()
    y0 = ops.dwconv_fwd(x, w, b, 1, 1, 2)
    y1 = ops.dwconv_fwd_fused(x, w, b, stride=1, dilation=1, pad=2)
    assert torch.equal(y0, y1)


def test_prologue_padding_is_zero_on_device():
    """x = 0 with a prologue shift of 1: every in-bounds tap sees 1, padding 0,
    so a box filter counts the in-bounds taps (exact in every dtype)."""
    from depthwise_convolution_gb300 import ops
    for dt, (H, W) in (("bf16", (12, 40)), ("fp32", (9, 9)), ("fp16", (6, 6))):
        tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dt]
        x = torch.zeros(1, H, W, 32, dtype=tdt, device="cuda")
        w = torch.ones(3, 3, 32, dtype=tdt, device="cuda")
        y = ops.dwconv_fwd_fused(x, w, in_shift=torch.ones(32, device="cuda"), in_act="relu", pad=1)
        rows = torch.tensor([2.0] + [3.0] * (H - 2) + [2.0])
        cols = torch.tensor([2.0] + [3.0] * (W - 2) + [2.0])
        expect = (rows[:, None] * cols[None, :])[None, :, :, None].expand(1, H, W, 32)
        assert torch.equal(y.float().cpu(), expect), (dt, ops.dwconv_last_kernel())


@pytest.mark.parametrize("act", ["silu", "gelu", "relu", "relu6"])
@pytest.mark.parametrize("F", [1, 3])
def test_activation_accuracy_fp32(act, F):
    """The fp32 activations on their own (a filter that passes x through:
    1x1 on the direct kernel, the centre tap of a 3x3 on the tiled one), as
    epilogue and as prologue, against the float64 definitions: within
    1e-6 |v| + 1e-7 (SiLU with the fast exponential and reciprocal; GELU
    with Abramowitz & Stegun 7.1.26, |erf error| <= 1.5e-7)."""
    import numpy as np
    import oracle
    from depthwise_convolution_gb300 import ops
    C, H, W = 32, 48, 64
    v = torch.linspace(-14.0, 14.0, H * W * C, dtype=torch.float64).reshape(1, H, W, C)
    x = v.float().cuda()
    w = torch.zeros(F, F, C, device="cuda")
    w[F // 2, F // 2] = 1.0
    ref = oracle.activation(v.float().double().numpy(), act)
    bound = 1e-6 * np.abs(v.numpy()) + 1e-7
    for mode in ("post", "pre"):
        kw = {"out_act": act} if mode == "post" else {"in_act": act}
        y = ops.dwconv_fwd_fused(x, w, pad=F // 2, **kw)
        err = np.abs(y.double().cpu().numpy() - ref)
        assert np.all(err <= bound), (mode, ops.dwconv_last_kernel(), float((err - bound).max()))
