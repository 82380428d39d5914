"""Strip filters (1 x K, K x 1 and the 5 x 51 / 51 x 5 pairs of factorised
large kernels) against the oracle: forward and input gradient, element by
element, with the kernel family each one is meant to take.  Filters taller
than wide run on the large-filter kernels in a transposed view (rows and
columns exchange roles in the kernel, the tensors stay in place).
"""
from __future__ import annotations

import pytest

from depthwise_convolution_gb300 import ops
from depthwise_convolution_gb300 import synthetic as syn
from parity import check_dgrad, check_fused, check_fwd, random_inputs

pytestmark = pytest.mark.gpu

# (dtype, (N, H, W, C, FH, FW, S, D, P), family)
CASES = [
    ("bf16", (2, 24, 40, 16, 51, 5, 1, 1, (25, 2)), "tiled_mma_large"),   # tall, transposed
    ("fp16", (2, 40, 24, 24, 5, 51, 1, 1, (2, 25)), "tiled_mma_large"),   # wide
    ("bf16", (3, 12, 30, 16, 51, 5, 1, 1, (25, 2)), "tiled_large"),       # transposed map too narrow for MMA
    ("fp32", (2, 30, 20, 32, 51, 5, 1, 1, (25, 2)), "tiled_large"),       # tall, transposed
    ("fp32", (2, 20, 30, 32, 5, 51, 1, 1, (2, 25)), "tiled_large"),
    ("fp32", (2, 33, 17, 36, 31, 1, 1, 1, (15, 0)), "tiled_large"),       # K x 1, transposed
    ("bf16", (2, 17, 33, 40, 1, 31, 1, 1, (0, 15)), "tiled_large"),       # 1 x K
    ("fp16", (2, 40, 19, 8, 31, 1, 1, 1, (15, 0)), "tiled_large"),        # K x 1, 16-bit
    ("bf16", (1, 30, 26, 16, 9, 3, 1, 1, (4, 1)), "tiled_large"),         # 9 x 3, transposed
]


def _ids(c):
    dt, (N, H, W, C, FH, FW, S, D, P), fam = c
    return f"{dt}-{N}x{H}x{W}x{C}-{FH}x{FW}-p{P}-{fam}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_strip_forward(case):
    dt, shape, fam = case
    N, H, W, C, FH, FW, S, D, P = shape
    d = random_inputs(dt, N, H, W, C, FH, FW, S, D, P, seed=61)
    check_fwd(d, dt, S, D, P, what="strip-fwd")
    assert ops.dwconv_last_kernel() == fam


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_strip_input_gradient(case):
    dt, shape, fam = case
    N, H, W, C, FH, FW, S, D, P = shape
    d = random_inputs(dt, N, H, W, C, FH, FW, S, D, P, seed=67)
    check_dgrad(d, dt, S, D, P, what="strip-dgrad")
    assert ops.dwconv_last_kernel() == fam


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_tall_strip_fused(dt):
    """The fused forward pass in the transposed view: a prologue on the
    tensor-core kernel (16-bit), the epilogue on the CUDA-core one (fp32)."""
    N, H, W, C, FH, FW, S, D, P = 2, 26, 30, 16, 51, 5, 1, 1, (25, 2)
    d = random_inputs(dt, N, H, W, C, FH, FW, S, D, P, seed=71)
    s0, t0 = syn.make_affine(C, 3, "pre")
    s1, t1 = syn.make_affine(C, 4, "post")
    pre = (s0, t0, "relu") if dt == "bf16" else None
    kernel = check_fused(d, dt, S, D, P, pre=pre, post=(s1, t1, "silu"), what="strip-fused")
    assert kernel == ("tiled_mma_large" if dt == "bf16" else "tiled_large")
