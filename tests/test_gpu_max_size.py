"""Tensors of more than 2^31 elements: every pass must address each image
correctly once element offsets leave the 32-bit range.

The inputs are a seeded block of B images repeated along N (image n is block
image n % B), so the oracle checks sampled images -- the first, the one that
contains element 2^31, the last -- from the block alone.  An offset that
wrapped at 32 bits would read another position (2^31 elements is not a whole
number of images here, so the wrapped read lands inside a different image at
a shifted pixel) and fail the comparison.  For the weight gradient dy is zero
except on the first and the last image, so the exact result is those two
images' contribution.  Tolerances are those of the other parity tests.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from depthwise_convolution_gb300 import ops
from parity import compare, random_inputs, to64

pytestmark = pytest.mark.gpu

LIMIT = 2**31
B = 8  # images in the seeded block


def _repeat(t: torch.Tensor, N: int) -> torch.Tensor:
    reps = (N + B - 1) // B
    return t.repeat(reps, *([1] * (t.dim() - 1)))[:N]


def _sampled(N, per_image):
    return [0, LIMIT // per_image, N - 1]


def test_16bit_training_passes_beyond_2_31_elements():
    N, H, W, C, FH, FW, S, D, P = 7200, 56, 56, 96, 7, 7, 1, 1, 3
    per = H * W * C
    assert N * per > LIMIT and LIMIT % per != 0
    d = random_inputs("fp16", B, H, W, C, FH, FW, S, D, P, seed=91, bias=False)
    w = d["w"].cuda()
    imgs = _sampled(N, per)

    x = _repeat(d["x"].cuda(), N)
    y = ops.dwconv_fwd(x, w, None, S, D, P)
    assert ops.dwconv_last_kernel() == "tiled_mma_ring"
    ops.dwconv_check_device_errors()
    for n in imgs:
        ref, mag = oracle.fwd(to64(d["x"][n % B:n % B + 1]), to64(d["w"]), None, S, D, P)
        compare(to64(y[n:n + 1]), ref, mag, "fp16", True, f"fwd image {n}")
    del y

    dy = _repeat(d["dy"].cuda(), N)
    dx = ops.dwconv_bwd_data(dy, w, H, W, S, D, P)
    assert ops.dwconv_last_kernel() == "tiled_mma_ring"
    ops.dwconv_check_device_errors()
    for n in imgs:
        ref, mag = oracle.dgrad(to64(d["dy"][n % B:n % B + 1]), to64(d["w"]), H, W, S, D, P)
        compare(to64(dx[n:n + 1]), ref, mag, "fp16", True, f"dgrad image {n}")
    del dx

    dy.zero_()
    ends = [0, N - 1]
    for n in ends:
        dy[n] = d["dy"][n % B].cuda()
    dw = ops.dwconv_bwd_filter(x, dy, FH, FW, S, D, P)
    assert ops.dwconv_last_kernel() == "tiled_wgrad"
    ops.dwconv_check_device_errors()
    xs = np.concatenate([to64(d["x"][n % B:n % B + 1]) for n in ends])
    dys = np.concatenate([to64(d["dy"][n % B:n % B + 1]) for n in ends])
    ref, mag = oracle.wgrad(xs, dys, FH, FW, S, D, P)
    compare(to64(dw), ref, mag, "fp16", False, "wgrad, first and last image")


def test_fp32_forward_beyond_2_31_elements():
    N, H, W, C, FH, FW, S, D, P = 5352, 56, 56, 128, 7, 7, 1, 1, 3
    per = H * W * C
    assert N * per > LIMIT and LIMIT % per != 0
    d = random_inputs("fp32", B, H, W, C, FH, FW, S, D, P, seed=92)
    x = _repeat(d["x"].cuda(), N)
    y = ops.dwconv_fwd(x, d["w"].cuda(), d["bias"].cuda(), S, D, P)
    assert ops.dwconv_last_kernel() == "tiled_small"
    ops.dwconv_check_device_errors()
    for n in _sampled(N, per):
        ref, mag = oracle.fwd(to64(d["x"][n % B:n % B + 1]), to64(d["w"]), to64(d["bias"]), S, D, P)
        compare(to64(y[n:n + 1]), ref, mag, "fp32", False, f"fp32 fwd image {n}")


def test_int8_direct_forward_beyond_2_31_outputs():
    # 5 channels: rows are not whole 16-byte copies, so the direct kernel runs.
    N, H, W, C, FH, FW, S, D, P = 104864, 64, 64, 5, 3, 3, 1, 1, 1
    per = H * W * C
    assert N * per > LIMIT and LIMIT % per != 0
    d = random_inputs("int8", B, H, W, C, FH, FW, S, D, P, seed=93)
    x = _repeat(d["x"].cuda(), N)
    y = ops.dwconv_fwd(x, d["w"].cuda(), d["bias"].cuda(), S, D, P)
    assert ops.dwconv_last_kernel() == "direct_fwd"
    ops.dwconv_check_device_errors()
    for n in _sampled(N, per):
        ref, mag = oracle.fwd(to64(d["x"][n % B:n % B + 1]), to64(d["w"]), to64(d["bias"]), S, D, P)
        compare(to64(y[n:n + 1]), ref, mag, "int8", False, f"int8 fwd image {n}")
