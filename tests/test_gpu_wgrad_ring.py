"""Tensor-core weight gradient (tiled_mma_wgrad.cu) on batches large enough
that each CTA walks a range of several bands: ranges start and end inside an
image column, cross from one column (image, column tile) into the next, and
refill the x-row ring there.  Element by element against the oracle, plus
determinism of the fixed-order split reduction at such a size."""
from __future__ import annotations

import pytest
import torch

from depthwise_convolution_gb300 import ops
from parity import check_wgrad, random_inputs

pytestmark = pytest.mark.gpu

# (dtype, (N, H, W, C, FH, FW, S, D, P))
CASES = [
    # 3 channel tiles x 672 bands of 14 per column: ranges of ~7 bands cross columns.
    ("bf16", (48, 56, 56, 24, 13, 13, 1, 1, 6)),
    # 3 column tiles per row (the last 22 wide), a ragged last band (37 rows),
    # a (2, 3)-block accumulator shape.  (16-bit channel rows must be 16-byte
    # aligned for the tiled kernels, so channel tiles are always whole here.)
    ("fp16", (6, 37, 150, 24, 23, 9, 1, 1, (11, 4))),
    # The 31x31 instance (40-row ring) with ranges of 3 bands across columns.
    ("bf16", (64, 56, 56, 8, 31, 31, 1, 1, 15)),
    # A tall strip through the transposed view (kernel rows = the tensors'
    # columns), several bands per range.
    ("fp16", (24, 56, 56, 16, 31, 5, 1, 1, (15, 2))),
]


def _ids(c):
    dt, (N, H, W, C, FH, FW, S, D, P) = c
    return f"{dt}-{N}x{H}x{W}x{C}-{FH}x{FW}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_ring_ranges_across_columns(case):
    dt, (N, H, W, C, FH, FW, S, D, P) = case
    d = random_inputs(dt, N, H, W, C, FH, FW, S, D, P, seed=91 + N)
    check_wgrad(d, dt, S, D, P, what="wgrad-ring")
    assert ops.dwconv_last_kernel() == "tiled_mma_wgrad"


def test_ring_wgrad_is_deterministic_across_columns():
    N, H, W, C, FH, FW, S, D, P = 48, 56, 56, 24, 13, 13, 1, 1, 6
    d = random_inputs("bf16", N, H, W, C, FH, FW, S, D, P, seed=97)
    x, dy = d["x"].cuda(), d["dy"].cuda()
    a = ops.dwconv_bwd_filter(x, dy, FH, FW, S, D, P)
    b = ops.dwconv_bwd_filter(x, dy, FH, FW, S, D, P)
    assert ops.dwconv_last_kernel() == "tiled_mma_wgrad"
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
