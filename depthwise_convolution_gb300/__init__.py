"""Depthwise 2-D convolution on one GB300 (sm_103a).

The work is done by libdwconv.so (C ABI in include/dwconv.h, CUDA kernels in
csrc/); this package is its Python binding.  Importing the package does not
load the library; the first call does, and fails loudly if it is missing.
"""
from .ops import (dwconv_bwd_bias, dwconv_bwd_bias_workspace_size, dwconv_bwd_data, dwconv_bwd_filter,
                  dwconv_bwd_filter_static, dwconv_bwd_filter_workspace_size, dwconv_check_device_errors,
                  dwconv_fwd, dwconv_fwd_fused, dwconv_last_kernel, dwconv_launch_count, dwconv_output_size)
from ._lib import DwconvError
from .autograd import DepthwiseConv2d, DepthwiseConv2dFunction, depthwise_conv2d

__all__ = ["dwconv_fwd", "dwconv_fwd_fused", "dwconv_bwd_data", "dwconv_bwd_filter",
           "dwconv_bwd_filter_workspace_size", "dwconv_bwd_filter_static", "dwconv_bwd_bias",
           "dwconv_bwd_bias_workspace_size", "dwconv_output_size",
           "dwconv_launch_count", "dwconv_last_kernel", "dwconv_check_device_errors",
           "DwconvError", "depthwise_conv2d", "DepthwiseConv2d", "DepthwiseConv2dFunction"]
