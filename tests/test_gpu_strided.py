"""Stride-2, dilation-1 layers (the down-sampling depthwise layer; "Tiles, halos
and partial sums" works its halo example at stride 2): all three passes match
the oracle and run on the strided tiled kernels, not the direct ones."""
import pytest
import torch

from depthwise_convolution_gb300 import ops
from parity import check_dgrad, check_fwd, check_wgrad, random_inputs

pytestmark = pytest.mark.gpu

# (N, H, W, C, F, P): odd and even map sizes, paddings below, at and above
# F // 2 (even and odd), channel tails (40 = 32 + 8), several row and column tiles.
CASES = [
    (2, 16, 15, 40, 3, 1),
    (2, 17, 18, 32, 3, 0),
    (1, 33, 29, 64, 3, 2),
    (2, 20, 21, 40, 5, 2),
    (1, 19, 24, 32, 5, 1),
    (2, 23, 22, 48, 7, 3),
    (1, 30, 31, 32, 7, 4),
    (3, 9, 8, 16, 5, 2),
    (2, 4, 5, 32, 3, 1),
]


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_stride2_all_passes(dtype, case):
    N, H, W, C, F, P = case
    d = random_inputs(dtype, N, H, W, C, F, F, 2, 1, P, seed=300 + sum(case))
    check_fwd(d, dtype, 2, 1, P)
    assert ops.dwconv_last_kernel() == "strided_fwd"
    check_fwd(dict(d, bias=None), dtype, 2, 1, P, what="fwd-nobias")
    check_dgrad(d, dtype, 2, 1, P)
    assert ops.dwconv_last_kernel() == "strided_dgrad"
    check_wgrad(d, dtype, 2, 1, P)
    assert ops.dwconv_last_kernel() == "strided_wgrad"


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_stride2_padding_per_axis(dtype):
    N, H, W, C, F, P = 2, 21, 26, 32, 5, (1, 3)
    d = random_inputs(dtype, N, H, W, C, F, F, 2, 1, P, seed=41)
    check_fwd(d, dtype, 2, 1, P)
    assert ops.dwconv_last_kernel() == "strided_fwd"
    check_dgrad(d, dtype, 2, 1, P)
    assert ops.dwconv_last_kernel() == "strided_dgrad"
    check_wgrad(d, dtype, 2, 1, P)
    assert ops.dwconv_last_kernel() == "strided_wgrad"


def test_stride2_full_size_bf16_3x3():
    """The down-sampling layer x[128,56,56,96], 3x3, stride 2, pad 1: forward
    and input gradient on sampled images, weight gradient in full."""
    N, H, W, C, F, P = 128, 56, 56, 96, 3, 1
    d = random_inputs("bf16", N, H, W, C, F, F, 2, 1, P, seed=56)
    images = [0, 63, 127]
    check_fwd(d, "bf16", 2, 1, P, images=images)
    assert ops.dwconv_last_kernel() == "strided_fwd"
    check_dgrad(d, "bf16", 2, 1, P, images=images)
    assert ops.dwconv_last_kernel() == "strided_dgrad"
    check_wgrad(d, "bf16", 2, 1, P)
    assert ops.dwconv_last_kernel() == "strided_wgrad"


def test_stride2_wgrad_is_deterministic():
    d = random_inputs("fp16", 8, 28, 28, 64, 5, 5, 2, 1, 2, seed=8)
    x, dy = d["x"].cuda(), d["dy"].cuda()
    a = ops.dwconv_bwd_filter(x, dy, 5, 5, 2, 1, 2)
    b = ops.dwconv_bwd_filter(x, dy, 5, 5, 2, 1, 2)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_stride2_unaligned_channels_take_the_direct_kernel():
    """fp32 with C = 6: channel rows are not whole 16-byte copies."""
    d = random_inputs("fp32", 1, 10, 10, 6, 3, 3, 2, 1, 1, seed=9)
    check_fwd(d, "fp32", 2, 1, 1)
    assert ops.dwconv_last_kernel() == "direct_fwd"
