"""Python binding of the C ABI, one function per entry point, same names.

Argument marshalling only: shapes, dtypes and device pointers of PyTorch CUDA
tensors are passed to libdwconv, which does all of the work on the GPU.
PyTorch provides device memory (outputs and workspace are allocated with
torch.empty when the caller passes none) and the current CUDA stream.
"""
from __future__ import annotations

import contextlib
import ctypes

import torch

from . import _lib

_NULL_CTX = contextlib.nullcontext()
_L = None


def _ll():
    """The loaded library (fast path after the first call)."""
    global _L
    if _L is None:
        _L = _lib.load()
    return _L

_DTYPE = {torch.int8: _lib.INT8, torch.float32: _lib.FP32, torch.float16: _lib.FP16,
          torch.bfloat16: _lib.BF16}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPE[torch.float8_e4m3fn] = _lib.FP8_E4M3


def _y_dtype(x: torch.Tensor, dt: int):
    """Forward output dtype: int32 for int8 data, bf16 for FP8, else x's."""
    if dt == _lib.INT8:
        return torch.int32
    if dt == _lib.FP8_E4M3:
        return torch.bfloat16
    return x.dtype


def _code(t: torch.Tensor) -> int:
    try:
        return _DTYPE[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _dev(t: torch.Tensor, name: str, ndim: int, ref: torch.Tensor = None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if ref is not None and t.device != ref.device:
        raise ValueError(f"{name} must be on {ref.device}, like the input")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (channels-last dense layout)")
    return t.data_ptr()


def _on(t: torch.Tensor):
    """The library works on the current device: make t's device current for the call
    (the default stream is then that device's current stream).  No switch when it
    already is current."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("inputs must be CUDA tensors")
    if t.get_device() == torch.cuda.current_device():
        return _NULL_CTX
    return torch.cuda.device(t.device)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _pair(v, what):
    if isinstance(v, (tuple, list)):
        if len(v) != 2:
            raise ValueError(f"{what} must be an int or an (h, w) pair")
        return int(v[0]), int(v[1])
    return int(v), int(v)


def _axes(stride, dilation, pad):
    """stride, dilation, pad (each an int or an (h, w) pair) -> the six per-axis ints."""
    (sh, sw), (dh, dw), (ph, pw) = _pair(stride, "stride"), _pair(dilation, "dilation"), _pair(pad, "pad")
    return sh, sw, dh, dw, ph, pw


def _out_hw(H, W, FH, FW, stride, dilation, pad):
    """(OH, OW) for the wrappers' shape checks (the library validates again):
    floor((X + 2P - D(F-1) - 1)/S) + 1 per axis; invalid sizes go through
    dwconv_output_size, which raises the library's error."""
    (sh, sw), (dh, dw), (ph, pw) = _pair(stride, "stride"), _pair(dilation, "dilation"), _pair(pad, "pad")
    if min(H, W, FH, FW, sh, sw, dh, dw) <= 0 or min(ph, pw) < 0:
        return dwconv_output_size(H, W, FH, FW, stride, dilation, pad)
    oh = (H + 2 * ph - dh * (FH - 1) - 1) // sh + 1
    ow = (W + 2 * pw - dw * (FW - 1) - 1) // sw + 1
    if oh < 1 or ow < 1:
        return dwconv_output_size(H, W, FH, FW, stride, dilation, pad)
    return oh, ow


def dwconv_output_size(H, W, FH, FW, stride=1, dilation=1, pad=0):
    """(OH, OW) of the forward pass; raises DwconvError on invalid sizes.
    stride, dilation and pad: an int (both axes) or an (h, w) pair."""
    oh, ow = ctypes.c_int(0), ctypes.c_int(0)
    _lib.check(_ll().dwconv_output_size_2d(H, W, FH, FW, *_axes(stride, dilation, pad),
                                                  ctypes.byref(oh), ctypes.byref(ow)),
               "dwconv_output_size")
    return oh.value, ow.value


def dwconv_fwd(x, w, bias=None, stride=1, dilation=1, pad=0, out=None, stream=None):
    """y = DWC(x, w) + bias.  x [N,H,W,C], w [FH,FW,C], bias [C] (fp32, or int32
    for int8 data) or None; stride, dilation, pad: int or (h, w).  Returns
    y [N,OH,OW,C] (int32 for int8 data)."""
    N, H, W, C = x.shape
    FH, FW = w.shape[0], w.shape[1]
    dt = _code(x)
    if w.dtype != x.dtype or tuple(w.shape) != (FH, FW, C):
        raise ValueError("w must be [FH, FW, C] with x's dtype")
    bias_dtype = torch.int32 if dt == _lib.INT8 else torch.float32
    if bias is not None and (bias.dtype != bias_dtype or tuple(bias.shape) != (C,)):
        raise ValueError(f"bias must be [C] {bias_dtype}")
    OH, OW = _out_hw(H, W, FH, FW, stride, dilation, pad)
    y_dtype = _y_dtype(x, dt)
    if out is None:
        out = torch.empty((N, OH, OW, C), dtype=y_dtype, device=x.device)
    elif out.dtype != y_dtype or tuple(out.shape) != (N, OH, OW, C):
        raise ValueError("out has the wrong shape or dtype")
    with _on(x):
        _lib.check(_ll().dwconv_fwd_2d(
            N, H, W, C, FH, FW, *_axes(stride, dilation, pad), dt,
            _dev(x, "x", 4), _dev(w, "w", 3, x), None if bias is None else _dev(bias, "bias", 1, x),
            _dev(out, "out", 4, x), _stream(stream)), "dwconv_fwd")
    return out


def _act(a) -> int:
    if isinstance(a, str):
        try:
            return _lib.ACTIVATIONS[a]
        except KeyError:
            raise ValueError(f"unknown activation {a!r}; one of {sorted(_lib.ACTIVATIONS)}") from None
    return int(a)


def _vec(v, C, name, ref):
    if v is None:
        return None
    if v.dtype != torch.float32 or tuple(v.shape) != (C,):
        raise ValueError(f"{name} must be [C] float32")
    return _dev(v, name, 1, ref)


def dwconv_fwd_fused(x, w, bias=None, in_scale=None, in_shift=None, in_act="none", out_scale=None,
                     out_shift=None, out_act="none", stride=1, dilation=1, pad=0, out=None, stream=None):
    """Forward pass with a BN+Act prologue and an affine+activation epilogue:
    x' = act_in(in_scale * x + in_shift) rounded to x's dtype (padding of x'
    is zero), y = act_out(out_scale * (DWC(x', w) + bias) + out_shift).
    Scales and shifts: [C] float32 CUDA tensors or None (1 and 0); activations:
    "none", "relu", "relu6", "silu", "gelu" (or the ABI codes).  A BatchNorm in
    inference form folds into scale = gamma / sqrt(var + eps) and
    shift = beta - mean * scale.  Other arguments as dwconv_fwd."""
    N, H, W, C = x.shape
    FH, FW = w.shape[0], w.shape[1]
    dt = _code(x)
    ia, oa = _act(in_act), _act(out_act)
    for v, name in ((in_scale, "in_scale"), (in_shift, "in_shift"), (out_scale, "out_scale"),
                    (out_shift, "out_shift"), (bias, "bias")):
        if v is not None and (v.dtype != torch.float32 or tuple(v.shape) != (C,)):
            raise ValueError(f"{name} must be [C] float32")
    if w.dtype != x.dtype or tuple(w.shape) != (FH, FW, C):
        raise ValueError("w must be [FH, FW, C] with x's dtype")
    OH, OW = _out_hw(H, W, FH, FW, stride, dilation, pad)
    y_dtype = _y_dtype(x, dt)
    if out is None:
        out = torch.empty((N, OH, OW, C), dtype=y_dtype, device=x.device)
    elif out.dtype != y_dtype or tuple(out.shape) != (N, OH, OW, C):
        raise ValueError("out has the wrong shape or dtype")
    with _on(x):
        _lib.check(_ll().dwconv_fwd_fused_2d(
            N, H, W, C, FH, FW, *_axes(stride, dilation, pad), dt,
            _dev(x, "x", 4), _vec(in_scale, C, "in_scale", x), _vec(in_shift, C, "in_shift", x), ia,
            _dev(w, "w", 3, x), None if bias is None else _dev(bias, "bias", 1, x),
            _vec(out_scale, C, "out_scale", x), _vec(out_shift, C, "out_shift", x), oa,
            _dev(out, "out", 4, x), _stream(stream)), "dwconv_fwd_fused")
    return out


def dwconv_bwd_data(dy, w, H, W, stride=1, dilation=1, pad=0, out=None, stream=None):
    """dx [N,H,W,C] from dy [N,OH,OW,C] and w [FH,FW,C]; stride, dilation, pad: int or (h, w)."""
    N, OH, OW, C = dy.shape
    FH, FW = w.shape[0], w.shape[1]
    dt = _code(dy)
    if w.dtype != dy.dtype or tuple(w.shape) != (FH, FW, C):
        raise ValueError("w must be [FH, FW, C] with dy's dtype")
    if _out_hw(H, W, FH, FW, stride, dilation, pad) != (OH, OW):
        raise ValueError("dy's spatial size is not the forward output of an H x W input")
    if out is None:
        out = torch.empty((N, H, W, C), dtype=dy.dtype, device=dy.device)
    elif out.dtype != dy.dtype or tuple(out.shape) != (N, H, W, C):
        raise ValueError("out has the wrong shape or dtype")
    with _on(dy):
        _lib.check(_ll().dwconv_bwd_data_2d(
            N, H, W, C, FH, FW, *_axes(stride, dilation, pad), dt,
            _dev(dy, "dy", 4), _dev(w, "w", 3, dy), _dev(out, "out", 4, dy), _stream(stream)),
            "dwconv_bwd_data")
    return out


def dwconv_bwd_filter_workspace_size(N, H, W, C, FH, FW, stride, dilation, pad, dtype) -> int:
    """Workspace bytes dwconv_bwd_filter needs (dtype: a torch dtype or ABI code)."""
    code = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(_ll().dwconv_bwd_filter_workspace_size_2d(N, H, W, C, FH, FW,
                                                               *_axes(stride, dilation, pad), code))


def dwconv_bwd_filter(x, dy, FH, FW, stride=1, dilation=1, pad=0, out=None, workspace=None,
                      stream=None, half_accumulate=False):
    """dw [FH,FW,C] fp32 from x [N,H,W,C] and dy [N,OH,OW,C].  half_accumulate
    (fp16 data only) calls dwconv_bwd_filter_ha: fp16 partial sums over short
    sub-units, merged in fp32 (an opt-in with a looser error bound)."""
    N, H, W, C = x.shape
    dt = _code(x)
    if dy.dtype != x.dtype:
        raise ValueError("dy must have x's dtype")
    if (dy.shape[0], dy.shape[3]) != (N, C) or \
            _out_hw(H, W, FH, FW, stride, dilation, pad) != tuple(dy.shape[1:3]):
        raise ValueError("dy's shape is not the forward output's")
    if out is None:
        out = torch.empty((FH, FW, C), dtype=torch.float32, device=x.device)
    elif out.dtype != torch.float32 or tuple(out.shape) != (FH, FW, C):
        raise ValueError("out must be [FH, FW, C] float32")
    if workspace is None:
        need = dwconv_bwd_filter_workspace_size(N, H, W, C, FH, FW, stride, dilation, pad, dt)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    fn = _ll().dwconv_bwd_filter_ha_2d if half_accumulate else _ll().dwconv_bwd_filter_2d
    with _on(x):
        _lib.check(fn(
            N, H, W, C, FH, FW, *_axes(stride, dilation, pad), dt,
            _dev(x, "x", 4), _dev(dy, "dy", 4, x), _dev(out, "out", 3, x),
            _dev(workspace, "workspace", workspace.dim(), x), ws_bytes, _stream(stream)),
            "dwconv_bwd_filter_ha" if half_accumulate else "dwconv_bwd_filter")
    return out


def dwconv_bwd_bias_workspace_size(N, OH, OW, C) -> int:
    return int(_ll().dwconv_bwd_bias_workspace_size(N, OH, OW, C))


def dwconv_bwd_bias(dy, out=None, workspace=None, stream=None):
    """db [C] fp32 = the sum of dy [N,OH,OW,C] over N, OH, OW."""
    N, OH, OW, C = dy.shape
    dt = _code(dy)
    if out is None:
        out = torch.empty((C,), dtype=torch.float32, device=dy.device)
    elif out.dtype != torch.float32 or tuple(out.shape) != (C,):
        raise ValueError("out must be [C] float32")
    need = dwconv_bwd_bias_workspace_size(N, OH, OW, C)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dy.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on(dy):
        _lib.check(_ll().dwconv_bwd_bias(
            N, OH, OW, C, dt, _dev(dy, "dy", 4), _dev(out, "out", 1, dy),
            _dev(workspace, "workspace", workspace.dim(), dy), ws_bytes, _stream(stream)), "dwconv_bwd_bias")
    return out


def dwconv_bwd_filter_static(x, dy, FH, FW, stride=1, dilation=1, pad=0, out=None, stream=None):
    """dw [FH,FW,C] fp32 like dwconv_bwd_filter, for callers that cannot allocate
    scratch: the library's built-in scratch array is used instead of a workspace.
    Only ``out`` is allocated here when the caller passes none."""
    N, H, W, C = x.shape
    dt = _code(x)
    if dy.dtype != x.dtype:
        raise ValueError("dy must have x's dtype")
    if (dy.shape[0], dy.shape[3]) != (N, C) or \
            _out_hw(H, W, FH, FW, stride, dilation, pad) != tuple(dy.shape[1:3]):
        raise ValueError("dy's shape is not the forward output's")
    if out is None:
        out = torch.empty((FH, FW, C), dtype=torch.float32, device=x.device)
    elif out.dtype != torch.float32 or tuple(out.shape) != (FH, FW, C):
        raise ValueError("out must be [FH, FW, C] float32")
    with _on(x):
        _lib.check(_ll().dwconv_bwd_filter_static(
            N, H, W, C, FH, FW, stride, dilation, pad, dt,
            _dev(x, "x", 4), _dev(dy, "dy", 4, x), _dev(out, "out", 3, x), _stream(stream)),
            "dwconv_bwd_filter_static")
    return out


def dwconv_check_device_errors(stream=None) -> None:
    """Wait for the stream; raise DwconvError if a library kernel gave up a bounded wait."""
    _lib.check(_ll().dwconv_check_device_errors(_stream(stream)), "dwconv_check_device_errors")


def dwconv_selftest_timeout(stream=None) -> None:
    """Enqueue the library's failure-detection self-test: a bounded wait that
    runs out (no fault, no hang); the next dwconv_check_device_errors raises
    DwconvError with DWCONV_ERR_TIMEOUT."""
    _lib.check(_ll().dwconv_selftest_timeout(_stream(stream)), "dwconv_selftest_timeout")


def dwconv_launch_count() -> int:
    """Kernels libdwconv has launched in this process."""
    return int(_ll().dwconv_launch_count())


def dwconv_last_kernel() -> str:
    """Kernel family of the latest pass launched from this thread."""
    return _ll().dwconv_last_kernel().decode()
