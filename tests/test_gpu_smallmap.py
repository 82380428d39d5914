"""7x7 maps with "same" padding (the last stage of the CNNs the Flash-DWC
evaluation runs): every pass matches the oracle; the forward pass and the
input gradient run on the whole-map kernel, which only issues the taps that
land inside the map (and so does the fp32 weight gradient)."""
import pytest
import torch

from depthwise_convolution_gb300 import ops
from parity import check_dbias, check_dgrad, check_fwd, check_wgrad, random_inputs

pytestmark = pytest.mark.gpu

# (N, C, F): image counts that are not a multiple of the 4 images per CTA,
# channel counts that leave lanes idle (40 = 20 pairs), several channel groups.
CASES = [(5, 40, 7), (8, 128, 7), (3, 64, 5), (9, 96, 3), (1, 16, 7), (6, 200, 5)]


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_smallmap_all_passes(dtype, case):
    N, C, F = case
    P = F // 2
    d = random_inputs(dtype, N, 7, 7, C, F, F, 1, 1, P, seed=700 + N + C + F)
    check_fwd(d, dtype, 1, 1, P)
    assert ops.dwconv_last_kernel() == "smallmap"
    check_fwd(dict(d, bias=None), dtype, 1, 1, P, what="fwd-nobias")
    check_dgrad(d, dtype, 1, 1, P)
    assert ops.dwconv_last_kernel() == "smallmap"
    check_wgrad(d, dtype, 1, 1, P)
    # fp32 on the whole-map weight gradient; 16-bit data on the register-tiled one
    assert ops.dwconv_last_kernel() == ("smallmap_wgrad" if dtype == "fp32" else "tiled_wgrad")
    check_dbias(d, dtype)


def test_smallmap_full_size_stage():
    """The bf16 stage x[128,7,7,768], 7x7: all images, all passes."""
    d = random_inputs("bf16", 128, 7, 7, 768, 7, 7, 1, 1, 3, seed=77)
    check_fwd(d, "bf16", 1, 1, 3)
    check_dgrad(d, "bf16", 1, 1, 3)
    check_wgrad(d, "bf16", 1, 1, 3)
    assert ops.dwconv_last_kernel() == "tiled_wgrad"


def test_smallmap_wgrad_is_deterministic():
    d = random_inputs("fp32", 16, 7, 7, 256, 7, 7, 1, 1, 3, seed=78)
    x, dy = d["x"].cuda(), d["dy"].cuda()
    a = ops.dwconv_bwd_filter(x, dy, 7, 7, 1, 1, 3)
    b = ops.dwconv_bwd_filter(x, dy, 7, 7, 1, 1, 3)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_other_padding_stays_on_the_tile_kernel():
    d = random_inputs("bf16", 2, 7, 7, 64, 7, 7, 1, 1, 2, seed=79)
    check_fwd(d, "bf16", 1, 1, 2)
    assert ops.dwconv_last_kernel() == "tiled_small"
