"""Autograd wrapper: depthwise 2-D convolution as a differentiable PyTorch op.

Tensors are channels-last and dense: x [N, H, W, C], w [FH, FW, C], bias [C]
(float32, or int32 for int8 data), y [N, OH, OW, C].  The forward pass calls
``dwconv_fwd``; the backward pass calls ``dwconv_bwd_data`` for dx,
``dwconv_bwd_filter`` for dw (float32, cast to w's dtype) and
``dwconv_bwd_bias`` for db.  This module only marshals arguments; every pass
runs in the library's kernels.  int8 data is forward only.
"""
from __future__ import annotations

import math

import torch

from . import ops


class DepthwiseConv2dFunction(torch.autograd.Function):
    """y = DWC(x, w) + bias with the library's three training passes."""

    @staticmethod
    def forward(ctx, x, w, bias, stride, dilation, pad, half_accumulate=False):
        x, w = x.contiguous(), w.contiguous()
        ctx.save_for_backward(x, w)
        ctx.conv = (stride, dilation, pad)
        ctx.half_accumulate = half_accumulate
        ctx.bias_dtype = None if bias is None else bias.dtype
        return ops.dwconv_fwd(x, w, None if bias is None else bias.contiguous(), stride, dilation, pad)

    @staticmethod
    def backward(ctx, dy):
        x, w = ctx.saved_tensors
        stride, dilation, pad = ctx.conv
        dy = dy.contiguous().to(x.dtype)
        dx = dw = db = None
        if ctx.needs_input_grad[0]:
            dx = ops.dwconv_bwd_data(dy, w, x.shape[1], x.shape[2], stride, dilation, pad)
        if ctx.needs_input_grad[1]:
            dw = ops.dwconv_bwd_filter(x, dy, w.shape[0], w.shape[1], stride, dilation, pad,
                                       half_accumulate=ctx.half_accumulate).to(w.dtype)
        if ctx.bias_dtype is not None and ctx.needs_input_grad[2]:
            db = ops.dwconv_bwd_bias(dy).to(ctx.bias_dtype)
        return dx, dw, db, None, None, None, None


def depthwise_conv2d(x, w, bias=None, stride=1, dilation=1, pad=0, half_accumulate=False):
    """Differentiable depthwise convolution on NHWC tensors (see the module docstring).
    stride, dilation, pad: int or (h, w).  half_accumulate (fp16 only) selects the
    opt-in hybrid-accumulation weight gradient."""
    return DepthwiseConv2dFunction.apply(x, w, bias, stride, dilation, pad, half_accumulate)


class DepthwiseConv2d(torch.nn.Module):
    """Depthwise convolution layer holding w [FH, FW, C] and an optional float32 bias.

    ``padding`` defaults to "same" for odd filters at stride 1, per axis:
    (dilation_h * (FH - 1) // 2, dilation_w * (FW - 1) // 2), so strip filters
    (1 x K, K x 1) keep the map size.  Weights are drawn from N(0, 1/(FH*FW)).
    """

    def __init__(self, channels, kernel_size, stride=1, dilation=1, padding=None, bias=True,
                 dtype=torch.bfloat16, device="cuda", half_accumulate=False):
        super().__init__()
        if isinstance(kernel_size, int):
            kernel_size = (kernel_size, kernel_size)
        FH, FW = kernel_size
        self.stride, self.dilation = stride, dilation
        self.half_accumulate = half_accumulate
        dh, dw = (dilation, dilation) if isinstance(dilation, int) else tuple(dilation)
        self.padding = (dh * (FH - 1) // 2, dw * (FW - 1) // 2) if padding is None else padding
        w = torch.randn(FH, FW, channels, device=device, dtype=torch.float32) / math.sqrt(FH * FW)
        self.weight = torch.nn.Parameter(w.to(dtype))
        self.bias = torch.nn.Parameter(torch.zeros(channels, device=device, dtype=torch.float32)) if bias else None

    def forward(self, x):
        return depthwise_conv2d(x, self.weight, self.bias, self.stride, self.dilation, self.padding,
                                self.half_accumulate)

    def extra_repr(self):
        FH, FW, C = self.weight.shape
        return (f"channels={C}, kernel_size=({FH}, {FW}), stride={self.stride}, dilation={self.dilation}, "
                f"padding={self.padding}, bias={self.bias is not None}")
