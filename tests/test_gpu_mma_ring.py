"""Warp-specialised tensor-core forward pass and input gradient
(tiled_mma_ring_kernel.cuh, 16-bit 5x5 and 7x7 on maps wider than 32
columns): CTA unit ranges that start and end inside a column of row bands,
cross into the next column (image, column tile or channel tile) and refill the
row ring there; columns of one band (every unit refills); ragged last bands and
column tiles; channel tails; more CTAs than units.  Element by element against
the oracle."""
from __future__ import annotations

import pytest
import torch

from depthwise_convolution_gb300 import ops
from parity import check_dgrad, check_fwd, random_inputs

pytestmark = pytest.mark.gpu

# (dtype, (N, H, W, C, FH, FW, S, D, P))
CASES = [
    # 24 columns of 7 bands over every SM: ranges of one or two units.
    ("bf16", (24, 56, 56, 32, 7, 7, 1, 1, 3)),
    # 96 x 2 columns of 5 bands (the last one row high), 40 of 64 columns
    # used: ranges of ~6 units across columns and channel tiles.
    ("fp16", (96, 33, 40, 64, 5, 5, 1, 1, 2)),
    # 3 column tiles (the last 22 wide), a channel tail (40 = 32 + 8).
    ("bf16", (6, 20, 150, 40, 5, 5, 1, 1, 2)),
    # Columns of one band: every unit loads both of its pieces.
    ("fp16", (40, 8, 64, 32, 7, 7, 1, 1, 3)),
    # No padding, 300 units: ranges of 2 units, output 24 x 64.
    ("bf16", (25, 30, 70, 128, 7, 7, 1, 1, 0)),
    # More input rows than one piece's halo: 5x5 with padding 0 on 9-row maps.
    ("fp16", (7, 9, 37, 32, 5, 5, 1, 1, 0)),
]


def _ids(c):
    dt, (N, H, W, C, FH, FW, S, D, P) = c
    return f"{dt}-{N}x{H}x{W}x{C}-{FH}x{FW}-p{P}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_ring_forward(case):
    dt, (N, H, W, C, FH, FW, S, D, P) = case
    d = random_inputs(dt, N, H, W, C, FH, FW, S, D, P, seed=131 + N)
    check_fwd(d, dt, S, D, P, what="fwd-ring")
    assert ops.dwconv_last_kernel() == "tiled_mma_ring"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_ring_input_gradient(case):
    dt, (N, H, W, C, FH, FW, S, D, P) = case
    d = random_inputs(dt, N, H, W, C, FH, FW, S, D, P, seed=137 + N)
    check_dgrad(d, dt, S, D, P, what="dgrad-ring")
    assert ops.dwconv_last_kernel() == "tiled_mma_ring"


def test_ring_forward_is_deterministic():
    N, H, W, C, FH, FW, S, D, P = 24, 56, 56, 64, 7, 7, 1, 1, 3
    d = random_inputs("bf16", N, H, W, C, FH, FW, S, D, P, seed=139)
    x, w = d["x"].cuda(), d["w"].cuda()
    a = ops.dwconv_fwd(x, w, None, S, D, P)
    b = ops.dwconv_fwd(x, w, None, S, D, P)
    ops.dwconv_check_device_errors()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
