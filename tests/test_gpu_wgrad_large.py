"""Weight gradient of large and strip filters -- 16-bit data on the
tensor-core kernel (tiled_mma_wgrad.cu), fp32 on the tiled tap-group kernel
(tiled_wgrad_large.cu) -- against the oracle, element by element within the
stated fp32-accumulation bounds, and bit-identical from call to call.
"""
from __future__ import annotations

import pytest
import torch

from depthwise_convolution_gb300 import ops
from parity import check_wgrad, random_inputs

pytestmark = pytest.mark.gpu

# (dtype, (N, H, W, C, FH, FW, S, D, P))
CASES = [
    ("bf16", (2, 20, 24, 40, 31, 31, 1, 1, 15)),   # several tap groups, channel tail
    ("fp32", (2, 19, 23, 36, 13, 13, 1, 1, 6)),
    ("fp16", (3, 30, 14, 16, 51, 5, 1, 1, (25, 2))),  # tall strip: transposed
    ("fp32", (2, 14, 30, 32, 5, 51, 1, 1, (2, 25))),
    ("bf16", (2, 17, 21, 24, 9, 9, 1, 1, 4)),
    ("fp32", (2, 33, 9, 8, 31, 1, 1, 1, (15, 0))),     # K x 1
    ("bf16", (1, 9, 33, 16, 1, 31, 1, 1, (0, 15))),    # 1 x K
    ("fp16", (2, 24, 24, 16, 9, 9, 2, 2, 8)),          # stride 2 dilation 2: even sub-grid
    ("fp32", (2, 12, 13, 12, 5, 3, 1, 1, (2, 1))),     # small non-square: no tiled_wgrad instance
    ("bf16", (2, 40, 70, 16, 13, 13, 1, 1, 6)),        # several dy tiles per row
    ("fp16", (2, 21, 19, 8, 17, 29, 1, 1, (8, 14))),   # 2 x 4 blocks, ragged both ways
    ("bf16", (1, 5, 6, 8, 11, 11, 1, 1, 5)),           # map smaller than the filter
]


def _ids(c):
    dt, (N, H, W, C, FH, FW, S, D, P) = c
    return f"{dt}-{N}x{H}x{W}x{C}-{FH}x{FW}-s{S}d{D}p{P}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_large_filter_wgrad(case):
    dt, (N, H, W, C, FH, FW, S, D, P) = case
    d = random_inputs(dt, N, H, W, C, FH, FW, S, D, P, seed=73)
    check_wgrad(d, dt, S, D, P, what="wgrad-large")
    assert ops.dwconv_last_kernel() == ("tiled_wgrad_large" if dt == "fp32" else "tiled_mma_wgrad")


def test_large_filter_wgrad_is_deterministic():
    N, H, W, C, FH, FW, S, D, P = 4, 28, 28, 64, 31, 31, 1, 1, 15
    d = random_inputs("bf16", N, H, W, C, FH, FW, S, D, P, seed=79)
    x, dy = d["x"].cuda(), d["dy"].cuda()
    a = ops.dwconv_bwd_filter(x, dy, FH, FW, S, D, P)
    b = ops.dwconv_bwd_filter(x, dy, FH, FW, S, D, P)
    assert ops.dwconv_last_kernel() == "tiled_mma_wgrad"
    assert torch.equal(a, b)
