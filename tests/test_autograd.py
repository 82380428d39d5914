"""The autograd wrapper: its gradients are the library's passes, and agree with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from depthwise_convolution_gb300 import DepthwiseConv2d, depthwise_conv2d, ops
from parity import compare, random_inputs, to64


def test_cpu_tensors_are_rejected():
    x = torch.zeros(1, 4, 4, 8, dtype=torch.bfloat16)
    w = torch.zeros(3, 3, 8, dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError)):
        depthwise_conv2d(x, w, None, 1, 1, 1)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,case", [
    ("bf16", (2, 20, 22, 64, 7, 7, 1, 1, 3)),
    ("fp16", (3, 14, 14, 32, 3, 3, 1, 1, 1)),
    ("fp32", (2, 12, 13, 16, 5, 5, 2, 2, 4)),
    ("bf16", (1, 24, 24, 16, 31, 31, 1, 1, 15)),
])
def test_gradients_are_the_library_passes(dtype, case):
    N, H, W, C, FH, FW, S, D, P = case
    d = random_inputs(dtype, N, H, W, C, FH, FW, S, D, P, seed=21)
    x = d["x"].cuda().requires_grad_()
    w = d["w"].cuda().requires_grad_()
    b = d["bias"].cuda().requires_grad_()
    dy = d["dy"].cuda()
    y = depthwise_conv2d(x, w, b, S, D, P)
    assert torch.equal(y, ops.dwconv_fwd(x.detach(), w.detach(), b.detach(), S, D, P))
    y.backward(dy)
    assert torch.equal(x.grad, ops.dwconv_bwd_data(dy, w.detach(), H, W, S, D, P))
    assert torch.equal(w.grad, ops.dwconv_bwd_filter(x.detach(), dy, FH, FW, S, D, P).to(w.dtype))
    assert torch.equal(b.grad, ops.dwconv_bwd_bias(dy))
    ref_db, mag_db = oracle.dbias(to64(d["dy"]))
    compare(to64(b.grad), ref_db, mag_db, dtype, False, "autograd db")
    ref_dx, mag_dx = oracle.dgrad(to64(d["dy"]), to64(d["w"]), H, W, S, D, P)
    compare(to64(x.grad), ref_dx, mag_dx, dtype, dtype != "fp32", "autograd dx")


@pytest.mark.gpu
def test_module_trains_one_step():
    torch.manual_seed(0)
    layer = DepthwiseConv2d(64, 7, dtype=torch.bfloat16)
    x = torch.randn(4, 16, 16, 64, device="cuda").to(torch.bfloat16)
    target = torch.randn(4, 16, 16, 64, device="cuda")
    opt = torch.optim.SGD(layer.parameters(), lr=0.1)
    loss0 = ((layer(x).float() - target) ** 2).mean()
    loss0.backward()
    opt.step()
    opt.zero_grad()
    loss1 = ((layer(x).float() - target) ** 2).mean()
    assert torch.isfinite(loss1) and loss1.item() < loss0.item()
    assert "kernel_size=(7, 7)" in repr(layer)


def test_module_same_padding_per_axis():
    layer = DepthwiseConv2d(16, (5, 51), dtype=torch.float32, device="cpu")
    assert layer.padding == (2, 25)
    assert DepthwiseConv2d(16, 7, dilation=2, dtype=torch.float32, device="cpu").padding == (6, 6)
    assert DepthwiseConv2d(16, 3, padding=0, dtype=torch.float32, device="cpu").padding == 0


@pytest.mark.gpu
def test_strip_layer_keeps_the_map_and_half_accumulate_flows_through():
    layer = DepthwiseConv2d(32, (51, 5), dtype=torch.float16)
    x = torch.randn(2, 30, 26, 32, device="cuda").to(torch.float16).requires_grad_()
    y = layer(x)
    assert y.shape == x.shape
    y.float().sum().backward()
    assert layer.weight.grad is not None and torch.isfinite(layer.weight.grad.float()).all()
    # the opt-in hybrid accumulation reaches the weight-gradient entry point (7x7 has the HA kernel)
    # (the backward pass runs on autograd's own thread: compare results, not the
    # thread-local kernel record)
    l7 = DepthwiseConv2d(32, 7, bias=False, dtype=torch.float16, half_accumulate=True)
    x7 = torch.randn(2, 20, 20, 32, device="cuda").to(torch.float16)
    y7 = l7(x7)
    dy7 = torch.randn_like(y7)
    y7.backward(dy7)
    w = l7.weight.detach()
    ha = ops.dwconv_bwd_filter(x7, dy7, 7, 7, 1, 1, 3, half_accumulate=True).to(w.dtype)
    exact = ops.dwconv_bwd_filter(x7, dy7, 7, 7, 1, 1, 3).to(w.dtype)
    assert torch.equal(l7.weight.grad, ha)
    assert not torch.equal(ha, exact)
