"""The seeded input generators (CPU): the same seed gives the same tensors, the
tensors of a workload are independent draws, the distributions and integer
ranges are the stated ones, and the workloads carry the benchmark shapes."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from depthwise_convolution_gb300 import synthetic as syn


def _wl(dtype="fp16", N=4, H=12, W=10, C=16, F=3, passes=("fwd", "dgrad", "wgrad"), seed=5, bias=True):
    return syn.Workload("t", dtype, N, H, W, C, F, F, 1, 1, F // 2, bias, passes, seed)


def test_same_seed_same_tensors_and_other_seed_other_tensors():
    a = syn.make_inputs(_wl(), dy_hw=(12, 10))
    b = syn.make_inputs(_wl(), dy_hw=(12, 10))
    c = syn.make_inputs(_wl(seed=6), dy_hw=(12, 10))
    for k in ("x", "w", "bias", "dy"):
        assert torch.equal(a[k], b[k])
        assert not torch.equal(a[k], c[k])


def test_tensors_of_a_workload_are_independent_draws():
    d = syn.make_inputs(_wl(N=8, H=16, W=16, C=32), dy_hw=(16, 16))
    x = d["x"].float().flatten().numpy()
    dy = d["dy"].float().flatten().numpy()
    assert x.shape == dy.shape and not np.array_equal(x, dy)
    assert abs(np.corrcoef(x, dy)[0, 1]) < 0.02


def test_normal_draws_have_the_stated_spread():
    wl = syn.Workload("t", "fp32", 64, 32, 32, 32, 7, 7, 1, 1, 3, True, ("fwd",), 2)
    d = syn.make_inputs(wl)
    x = d["x"].numpy().astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    w = d["w"].numpy().astype(np.float64)
    assert abs(w.std() * 7 - 1.0) < 0.1  # sigma = 1/7 from 1568 values (standard error ~2 %)
    b = d["bias"].numpy().astype(np.float64)
    assert d["bias"].dtype == torch.float32 and b.shape == (32,)
    big = syn.normal((1 << 20,), math.sqrt(0.1), 9, 2).astype(np.float64)
    assert abs(big.var() - 0.1) < 0.002


def test_sixteen_bit_inputs_are_the_rounded_float32_draws():
    wl = _wl("bf16")
    d = syn.make_inputs(wl, dy_hw=(12, 10))
    raw = syn.normal((wl.N, wl.H, wl.W, wl.C), 1.0, wl.seed, 0)
    assert d["x"].dtype == torch.bfloat16
    assert torch.equal(d["x"], torch.from_numpy(raw).to(torch.bfloat16))


def test_int8_ranges_are_inclusive():
    wl = syn.Workload("t", "int8", 8, 32, 32, 5, 3, 3, 1, 1, 1, True, ("fwd",), 1)
    d = syn.make_inputs(wl)
    x = d["x"].to(torch.int64)
    assert d["x"].dtype == torch.int8 and int(x.min()) == -128 and int(x.max()) == 127
    assert d["bias"].dtype == torch.int32 and d["dy"] is None
    v = syn.uniform_int((200000,), -1000, 1000, 3, 2)
    assert v.min() == -1000 and v.max() == 1000


def test_backward_workloads_need_the_output_size():
    with pytest.raises(ValueError, match="dy_hw"):
        syn.make_inputs(_wl())
    fwd_only = syn.make_inputs(_wl(passes=("fwd",)))
    assert fwd_only["dy"] is None


def test_chunked_generation_is_independent_of_the_tensor_size_it_sits_in():
    # The first rows of a tall tensor are the same draws as a short tensor with the same seed.
    short = syn.normal((3, 1000), 1.0, 4, 0)
    tall = syn.normal((50, 1000), 1.0, 4, 0)
    assert np.array_equal(short, tall[:3])


def test_affine_vectors_for_the_fused_pass():
    s0, t0 = syn.make_affine(4096, 3, "pre")
    s1, t1 = syn.make_affine(4096, 3, "post")
    assert s0.dtype == torch.float32 and s0.shape == (4096,)
    assert abs(float(s0.mean()) - 1.0) < 0.05 and abs(float(s0.std()) - 0.5) < 0.05
    assert abs(float(t0.mean())) < 0.05 and abs(float(t0.std()) - 0.5) < 0.05
    assert not torch.equal(s0, s1) and not torch.equal(t0, t1)


def test_benchmark_workloads_have_the_stated_shapes():
    wl = syn.WORKLOADS["fp16-train-7x7-128x56x56x96"]
    assert (wl.dtype, wl.N, wl.H, wl.W, wl.C, wl.FH, wl.FW, wl.stride, wl.dilation, wl.pad) == \
        ("fp16", 128, 56, 56, 96, 7, 7, 1, 1, 3)
    assert set(wl.passes) == {"fwd", "dgrad", "wgrad"} and not wl.bias
    big = syn.WORKLOADS["bf16-fwd-31x31-32x56x56x128"]
    assert (big.N, big.C, big.FH, big.FW, big.pad, big.bias) == (32, 128, 31, 31, 15, True)
    assert syn.WORKLOADS["int8-fwd-3x3-1x8x8x5"].C == 5
    s2 = syn.WORKLOADS["bf16-train-5x5s2d2-64x112x112x64"]
    assert (s2.stride, s2.dilation, s2.pad, s2.FH) == (2, 2, 4, 5)
