"""GPU parity: the CUDA path against the oracle, element by element, on the
same seeded, quantised inputs.  Small shapes that span several tiles with
ragged tails, edge cases, and the five workloads at full size (every element
of every pass)."""
import numpy as np
import pytest
import torch

import oracle
from depthwise_convolution_gb300 import DwconvError, ops, synthetic
from parity import (TORCH, check_dbias, check_dgrad, check_fwd, check_wgrad, compare, random_inputs, to64)

pytestmark = pytest.mark.gpu

# (N, H, W, C, FH, FW, S, D, P)
SMALL = [
    (2, 13, 11, 40, 3, 3, 1, 1, 1),      # 3x3, channel tail 40 = 32 + 8, ragged rows/columns
    (3, 23, 19, 64, 5, 5, 1, 1, 2),      # 5x5 over several tiles
    (2, 30, 29, 96, 7, 7, 1, 1, 3),      # 7x7 over several tiles and channel slabs
    (1, 9, 9, 32, 7, 7, 1, 1, 0),        # no padding
    (2, 20, 22, 32, 5, 5, 2, 2, 4),      # stride 2, dilation 2: even sub-grid
    (2, 21, 17, 48, 5, 5, 2, 2, 3),      # stride 2, dilation 2, odd pad: odd sub-grid
    (2, 16, 15, 24, 3, 3, 2, 1, 1),      # stride 2
    (2, 12, 12, 8, 3, 3, 1, 2, 2),       # dilation 2
    (1, 7, 7, 6, 4, 2, 1, 1, 1),         # non-square, even filter extent, C = 6
    (2, 10, 10, 5, 3, 3, 1, 1, 1),       # odd channel count
    (1, 40, 40, 32, 31, 31, 1, 1, 15),   # large filter
    (1, 5, 5, 16, 7, 7, 1, 1, 3),        # map smaller than the filter
    (4, 7, 7, 64, 7, 7, 1, 1, 3),        # 7x7 map: several images per CTA
    (3, 14, 14, 32, 7, 7, 1, 1, 3),      # 14x14 map
    (2, 1, 1, 16, 3, 3, 1, 1, 1),        # 1x1 map
    (1, 6, 6, 16, 3, 3, 3, 1, 1),        # stride 3
    (2, 9, 8, 16, 3, 5, 1, 1, 2),        # FH != FW on the tiled path (pads differ by axis)
    (1, 11, 11, 2, 3, 3, 1, 1, 1),       # C = 2
    (2, 20, 19, 40, 9, 13, 1, 1, 5),     # large-filter path, FH != FW, channel tail
    (1, 33, 30, 64, 11, 11, 2, 2, 10),   # large filter on the stride-2 dilation-2 sub-grid
    (3, 9, 30, 32, 15, 15, 1, 1, 7),     # large filter, map shorter than the filter
    (2, 24, 21, 40, 31, 31, 1, 1, 15),   # 31x31 tensor-core path on a narrow map, 5 channel tiles
    (1, 30, 45, 24, 13, 13, 1, 1, 6),    # 13x13 tensor-core path, ragged row band
    (2, 19, 20, 16, 13, 9, 1, 1, 4),     # FH != FW on the large tensor-core path
    (1, 41, 41, 16, 13, 13, 2, 2, 12),   # 13x13 on the stride-2 dilation-2 sub-grid
    (3, 30, 28, 32, 3, 3, 2, 2, 2),      # stride-2 dgrad on a narrow phase grid (two-image tiles)
    (2, 45, 43, 32, 7, 7, 2, 2, 5),      # stride-2 dgrad, odd sizes, phase 1
]


# (N, H, W, C, FH, FW, (sh, sw), (dh, dw), (ph, pw)): per-axis stride, dilation, padding
AXES = [
    (2, 9, 40, 32, 1, 31, 1, 1, (0, 15)),             # 1 x 31 strip, "same" padding
    (2, 40, 9, 32, 31, 1, 1, 1, (15, 0)),             # 31 x 1 strip
    (2, 20, 40, 32, 5, 51, 1, 1, (2, 25)),            # 5 x 51 strip (large-filter path)
    (2, 21, 30, 32, 3, 5, (2, 1), 1, (1, 2)),         # stride 2 along H only
    (2, 24, 26, 32, 7, 7, (2, 2), (2, 2), (3, 4)),    # s2 d2 with unequal padding: phases (1, 0)
    (1, 17, 33, 40, 5, 5, (1, 2), (2, 2), (4, 3)),    # stride 1 x 2, dilation 2: sub-grids differ by axis
    (2, 15, 19, 16, 3, 3, (3, 1), (1, 2), (0, 2)),    # direct path
]


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("case", AXES, ids=lambda c: "x".join(map(str, c)).replace(" ", ""))
def test_per_axis_parameters_all_passes(dtype, case):
    N, H, W, C, FH, FW, S, D, P = case
    d = random_inputs(dtype, N, H, W, C, FH, FW, S, D, P, seed=abs(hash(case)) % 1000 + 3)
    check_fwd(d, dtype, S, D, P)
    check_dgrad(d, dtype, S, D, P)
    check_wgrad(d, dtype, S, D, P)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c)))
def test_small_shapes_all_passes(dtype, case):
    N, H, W, C, FH, FW, S, D, P = case
    d = random_inputs(dtype, N, H, W, C, FH, FW, S, D, P, seed=hash(case) % 1000 + 7)
    check_fwd(d, dtype, S, D, P)
    d_nobias = dict(d, bias=None)
    check_fwd(d_nobias, dtype, S, D, P, what="fwd-nobias")
    check_dgrad(d, dtype, S, D, P)
    check_wgrad(d, dtype, S, D, P)
    check_dbias(d, dtype)


def test_int8_tail_channels_bit_exact():
    wl = synthetic.WORKLOADS["int8-fwd-3x3-1x8x8x5"]
    d = synthetic.make_inputs(wl)
    check_fwd(d, "int8", wl.stride, wl.dilation, wl.pad, what=wl.name)


@pytest.mark.parametrize("case", [(3, 9, 7, 13, 3, 3, 1, 1, 1), (1, 6, 6, 64, 5, 5, 2, 1, 2),
                                  (2, 8, 8, 7, 3, 3, 2, 2, 2)])
def test_int8_other_shapes_bit_exact(case):
    N, H, W, C, FH, FW, S, D, P = case
    d = random_inputs("int8", N, H, W, C, FH, FW, S, D, P, seed=99)
    check_fwd(d, "int8", S, D, P)


def test_int8_wraps_like_two_complement():
    """Sums beyond int32 wrap modulo 2^32 (documented behaviour)."""
    x = torch.full((1, 3, 3, 2), -128, dtype=torch.int8)
    w = torch.full((3, 3, 2), -128, dtype=torch.int8)
    b = torch.tensor([2**31 - 1, -2**31], dtype=torch.int32)
    y = ops.dwconv_fwd(x.cuda(), w.cuda(), b.cuda(), 1, 1, 1).cpu()
    ref, _ = oracle.fwd(to64(x), to64(w), to64(b), 1, 1, 1)
    compare(to64(y), ref, None, "int8", False, "wrap")


FULL = [wl for wl in synthetic.WORKLOADS.values() if wl.dtype != "int8"]


def full_inputs(wl):
    OH, OW = oracle.out_extent(wl.H, wl.FH, wl.stride, wl.dilation, wl.pad), \
        oracle.out_extent(wl.W, wl.FW, wl.stride, wl.dilation, wl.pad)
    return synthetic.make_inputs(wl, dy_hw=(OH, OW) if "dgrad" in wl.passes else None)


@pytest.mark.parametrize("wl", FULL, ids=lambda w: w.name)
def test_full_size_workloads(wl):
    d = full_inputs(wl)
    # Every image of the forward pass and the input gradient, every element.
    check_fwd(d, wl.dtype, wl.stride, wl.dilation, wl.pad, what=f"{wl.name} fwd")
    if "dgrad" in wl.passes:
        check_dgrad(d, wl.dtype, wl.stride, wl.dilation, wl.pad, what=f"{wl.name} dgrad")
    if "wgrad" in wl.passes:
        check_wgrad(d, wl.dtype, wl.stride, wl.dilation, wl.pad, what=f"{wl.name} wgrad")
        check_dbias(d, wl.dtype, what=f"{wl.name} dbias")


def test_dbias_is_deterministic_and_rejects_int8():
    d = random_inputs("fp16", 8, 28, 28, 96, 7, 7, 1, 1, 3, seed=6)
    dy = d["dy"].cuda()
    a, b = ops.dwconv_bwd_bias(dy), ops.dwconv_bwd_bias(dy)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    with pytest.raises(DwconvError):
        ops.dwconv_bwd_bias(torch.zeros(1, 2, 2, 4, dtype=torch.int8, device="cuda"))


def test_wgrad_is_deterministic():
    d = random_inputs("bf16", 4, 28, 28, 96, 7, 7, 1, 1, 3, seed=5)
    x, dy = d["x"].cuda(), d["dy"].cuda()
    a = ops.dwconv_bwd_filter(x, dy, 7, 7, 1, 1, 3)
    b = ops.dwconv_bwd_filter(x, dy, 7, 7, 1, 1, 3)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_side_stream_and_launch_count():
    d = random_inputs("fp16", 2, 16, 16, 32, 7, 7, 1, 1, 3, seed=3)
    s = torch.cuda.Stream()
    before = ops.dwconv_launch_count()
    with torch.cuda.stream(s):
        x, w = d["x"].cuda(), d["w"].cuda()
        y = ops.dwconv_fwd(x, w, None, 1, 1, 3, stream=s)
    s.synchronize()
    assert ops.dwconv_launch_count() > before
    ref, mag = oracle.fwd(to64(d["x"]), to64(d["w"]), None, 1, 1, 3)
    compare(to64(y), ref, mag, "fp16", True, "side stream")


def test_zero_input_gives_bias_only():
    x = torch.zeros(2, 9, 9, 32, dtype=torch.bfloat16, device="cuda")
    w = torch.randn(7, 7, 32, device="cuda").to(torch.bfloat16)
    b = torch.randn(32, device="cuda")
    y = ops.dwconv_fwd(x, w, b, 1, 1, 3)
    assert torch.equal(y.float(), b.to(torch.bfloat16).float().expand_as(y))


@pytest.mark.parametrize("dtype,case,pass_name,family", [
    ("fp16", (2, 40, 40, 32, 7, 7, 1, 1, 3), "fwd", "tiled_mma_ring"),
    ("bf16", (2, 40, 40, 32, 7, 7, 1, 1, 3), "dgrad", "tiled_mma_ring"),
    ("bf16", (2, 40, 40, 32, 3, 3, 1, 1, 1), "fwd", "tiled_mma"),
    ("fp16", (2, 30, 30, 32, 7, 7, 1, 1, 3), "fwd", "tiled_mma"),
    ("bf16", (1, 40, 40, 32, 31, 31, 1, 1, 15), "fwd", "tiled_mma_large"),
    ("fp32", (2, 40, 40, 32, 7, 7, 1, 1, 3), "fwd", "tiled_small"),
    ("fp32", (1, 30, 30, 32, 15, 15, 1, 1, 7), "fwd", "tiled_large"),
    ("bf16", (1, 30, 30, 32, 15, 15, 1, 1, 7), "fwd", "tiled_mma_large"),
    ("bf16", (2, 16, 15, 24, 3, 3, 2, 1, 1), "dgrad", "strided_dgrad"),
    ("fp16", (2, 40, 40, 32, 7, 7, 1, 1, 3), "wgrad", "tiled_wgrad"),
    ("bf16", (2, 10, 10, 5, 3, 3, 1, 1, 1), "fwd", "direct_fwd"),
])
def test_kernel_family_reported(dtype, case, pass_name, family):
    """The dispatch picks the intended kernel family, and says so."""
    N, H, W, C, FH, FW, S, D, P = case
    d = random_inputs(dtype, N, H, W, C, FH, FW, S, D, P, seed=11)
    x, w, dy = d["x"].cuda(), d["w"].cuda(), d["dy"].cuda()
    if pass_name == "fwd":
        ops.dwconv_fwd(x, w, None, S, D, P)
    elif pass_name == "dgrad":
        ops.dwconv_bwd_data(dy, w, H, W, S, D, P)
    else:
        ops.dwconv_bwd_filter(x, dy, FH, FW, S, D, P)
    torch.cuda.synchronize()
    assert ops.dwconv_last_kernel() == family


def test_tiled_path_from_a_fresh_thread():
    """A thread whose first CUDA work is a library call still gets the tiled
    kernels (tensor-map encoding needs a context bound in that thread)."""
    import threading
    d = random_inputs("bf16", 2, 20, 22, 64, 7, 7, 1, 1, 3, seed=4)
    dy, w = d["dy"].cuda(), d["w"].cuda()
    torch.cuda.synchronize()
    seen = {}

    def worker():
        dx = ops.dwconv_bwd_data(dy, w, 20, 22, 1, 1, 3)
        seen["kernel"] = ops.dwconv_last_kernel()
        torch.cuda.synchronize()
        seen["dx"] = dx

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert seen["kernel"] == "tiled_mma"
    assert torch.equal(seen["dx"], ops.dwconv_bwd_data(dy, w, 20, 22, 1, 1, 3))
