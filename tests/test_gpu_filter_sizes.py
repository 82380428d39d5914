"""The odd square filters the Flash-DWC evaluation sweeps (3 to 51, §6.1), in
fp16 and bf16: every pass matches the oracle, and each one runs on the kernel
family the dispatch intends for it -- the tensor-core Toeplitz kernels for the
large filters up to 31 x 31, the CUDA-core large-filter kernels beyond."""
import pytest
import torch

from depthwise_convolution_gb300 import ops
from parity import check_dgrad, check_fwd, check_wgrad, random_inputs

pytestmark = pytest.mark.gpu

SIZES = list(range(9, 32, 2)) + [51]


def families(F):
    """(fwd and dgrad family, wgrad family) expected for an F x F 16-bit filter."""
    if F <= 31:
        return "tiled_mma_large", "tiled_mma_wgrad"
    return "tiled_large", "tiled_wgrad_large"


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("F", SIZES)
def test_square_filter_family_and_parity(dtype, F):
    # 36 columns (> 32: the 64-column tile), 29 rows (a ragged row band), three
    # channel tiles of 8 with a tail, "same" padding.
    N, H, W, C, P = 2, 29, 36, 24, F // 2
    d = random_inputs(dtype, N, H, W, C, F, F, 1, 1, P, seed=1000 + F)
    fwd_family, wgrad_family = families(F)
    check_fwd(d, dtype, 1, 1, P, what=f"{F}x{F} fwd")
    assert ops.dwconv_last_kernel() == fwd_family
    check_dgrad(d, dtype, 1, 1, P, what=f"{F}x{F} dgrad")
    assert ops.dwconv_last_kernel() == fwd_family
    check_wgrad(d, dtype, 1, 1, P, what=f"{F}x{F} wgrad")
    assert ops.dwconv_last_kernel() == wgrad_family


@pytest.mark.parametrize("F", [9, 17, 27])
def test_square_filter_narrow_map(F):
    """Maps of 17 to 32 columns take the 32-column tile of the same kernel."""
    N, H, W, C, P = 2, 21, 24, 16, F // 2
    d = random_inputs("bf16", N, H, W, C, F, F, 1, 1, P, seed=2000 + F)
    check_fwd(d, "bf16", 1, 1, P, what=f"{F}x{F} narrow fwd")
    assert ops.dwconv_last_kernel() == "tiled_mma_large"
    check_dgrad(d, "bf16", 1, 1, P, what=f"{F}x{F} narrow dgrad")
    assert ops.dwconv_last_kernel() == "tiled_mma_large"


def test_non_square_filter_of_a_compiled_height():
    """A 21 x 15 filter: height 21 is compiled with two 16-input blocks, and a
    15-wide filter needs two as well."""
    N, H, W, C, P = 1, 30, 40, 16, (10, 7)
    d = random_inputs("fp16", N, H, W, C, 21, 15, 1, 1, P, seed=77)
    check_fwd(d, "fp16", 1, 1, P)
    assert ops.dwconv_last_kernel() == "tiled_mma_large"
    torch.cuda.synchronize()
