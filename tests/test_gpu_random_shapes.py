"""Seeded random shapes across dtypes, filter kinds (small, large, strips),
strides, dilations and paddings: every pass against the oracle, element by
element.  The shape of each case is a function of its seed (in the test id),
so a failure reproduces exactly."""
from __future__ import annotations

import random

import pytest

from depthwise_convolution_gb300 import ops
from parity import check_dgrad, check_fwd, check_wgrad, out_hw, random_inputs

pytestmark = pytest.mark.gpu


def draw(seed):
    rng = random.Random(seed)
    dtype = rng.choice(["fp32", "fp16", "bf16"])
    kind = rng.choice(["small", "small", "large", "strip"])
    if kind == "small":
        FH = FW = rng.choice([3, 5, 7])
    elif kind == "large":
        FH, FW = rng.randint(8, 31), rng.randint(8, 31)
    else:
        FH, FW = (rng.randint(9, 33), rng.randint(1, 5))
        if rng.random() < 0.5:
            FH, FW = FW, FH
    S = rng.choice([1, 1, 1, 2])
    D = rng.choice([1, 1, 2]) if kind == "small" else 1
    N = rng.randint(1, 6)
    H, W = rng.randint(1, 48), rng.randint(1, 72)
    C = 8 * rng.randint(1, 8) if rng.random() < 0.8 else rng.randint(1, 40)
    P = (rng.randint(0, D * (FH - 1)), rng.randint(0, D * (FW - 1)))
    return dtype, (N, H, W, C, FH, FW, S, D, P)


def valid(case):
    N, H, W, C, FH, FW, S, D, P = case
    OH, OW = out_hw(H, W, FH, FW, S, D, P)
    return OH >= 1 and OW >= 1


SEEDS = [s for s in range(400) if valid(draw(s)[1])][:96]


def _id(seed):
    dt, (N, H, W, C, FH, FW, S, D, P) = draw(seed)
    return f"{seed}-{dt}-{N}x{H}x{W}x{C}-{FH}x{FW}-s{S}d{D}p{P[0]},{P[1]}"


@pytest.mark.parametrize("seed", SEEDS, ids=_id)
def test_random_shape_all_passes(seed):
    dtype, (N, H, W, C, FH, FW, S, D, P) = draw(seed)
    d = random_inputs(dtype, N, H, W, C, FH, FW, S, D, P, seed=5000 + seed)
    check_fwd(d, dtype, S, D, P, what=f"{_id(seed)} fwd")
    check_dgrad(d, dtype, S, D, P, what=f"{_id(seed)} dgrad")
    check_wgrad(d, dtype, S, D, P, what=f"{_id(seed)} wgrad")
    assert ops.dwconv_last_kernel()
