"""FP8 E4M3 forward pass (x, w in E4M3, fp32 accumulation, bf16 output)
against the oracle, which decodes the E4M3 codes from their bits: the
16-bit-input bound 2e-3 * (sum |w x| + |b|) plus half an ulp of bf16."""
from __future__ import annotations

import pytest
import torch

from depthwise_convolution_gb300 import ops
from depthwise_convolution_gb300 import synthetic as syn
from parity import check_fused, check_fwd, random_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not hasattr(torch, "float8_e4m3fn"), reason="torch without float8_e4m3fn")]

CASES = [
    ((2, 19, 45, 48, 7, 7, 1, 1, 3), "tiled_mma"),      # tensor cores: G = 8, channel tail
    ((3, 22, 20, 32, 5, 5, 1, 1, 2), "tiled_mma"),      # G = 4
    ((2, 9, 12, 64, 3, 3, 1, 1, 1), "tiled_mma"),       # G = 2, two images per unit
    ((2, 24, 24, 16, 3, 3, 2, 2, 2), "tiled_mma"),      # stride 2 dilation 2: even sub-grid
    ((4, 7, 7, 64, 7, 7, 1, 1, 3), "tiled_small"),      # 7x7 maps: CUDA-core kernel
    ((2, 12, 15, 32, 3, 5, 1, 1, (1, 2)), "tiled_small"),
    ((2, 13, 13, 16, 3, 3, 2, 1, 1), "direct_fwd"),     # stride 2
    ((1, 9, 11, 8, 3, 3, 1, 1, 1), "direct_fwd"),       # C * 1 byte not a 16-byte row
    ((2, 17, 19, 32, 9, 9, 1, 1, 4), "direct_fwd"),     # filter without an FP8 tiled instance
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[0][:6])) + "-" + c[1])
def test_fp8_forward(case):
    (N, H, W, C, FH, FW, S, D, P), fam = case
    d = random_inputs("fp8", N, H, W, C, FH, FW, S, D, P, seed=83)
    check_fwd(d, "fp8", S, D, P, what="fp8-fwd")
    assert ops.dwconv_last_kernel() == fam


def test_fp8_full_size_sampled():
    """The 7x7 64x56x56x128 layer with E4M3 inputs, checked on sampled images."""
    d = random_inputs("fp8", 64, 56, 56, 128, 7, 7, 1, 1, 3, seed=89)
    check_fwd(d, "fp8", 1, 1, 3, images=[0, 17, 63], what="fp8-fwd-full")
    assert ops.dwconv_last_kernel() == "tiled_mma"


def test_fp8_dequantising_epilogue():
    """A per-channel dequantisation scale and a ReLU in the fused epilogue."""
    N, H, W, C, FH, FW, S, D, P = 2, 20, 26, 32, 7, 7, 1, 1, 3
    d = random_inputs("fp8", N, H, W, C, FH, FW, S, D, P, seed=97)
    s, t = syn.make_affine(C, 9, "post")
    kernel = check_fused(d, "fp8", S, D, P, post=(s.abs() * 0.01, t, "relu"), what="fp8-fused")
    assert kernel == "tiled_mma"
