"""Depthwise-convolution oracle: plain, slow, obviously correct CPU code.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The library
(``depthwise_convolution_gb300``) never imports it and shares no code with it.

Contents
--------
``fwd`` / ``dgrad`` / ``wgrad``
    The definition of the operator and of its two training passes written out
    as direct loops in C (``dwconv_oracle.c``), float64 for floating-point data
    and int64 for integer data, threaded over channel ranges.  Each returns the
    result and the per-element magnitude ``mag`` (sum of |products| plus |bias|)
    that the parity tolerance scales with.
``decode_e4m3``
    FP8 E4M3 codes to float64, from the format's bit definition.
``dbias``
    The adjoint of the bias term (sum of dy over n, oh, ow), in numpy.
``fwd_fused`` / ``prologue`` / ``activation`` / ``round_to``
    The forward pass with a BN+Act before it (x rounded back to its storage
    format, as the unfused layer stores it) and an affine map plus activation
    after it; ReLU, ReLU6, SiLU and GELU from their definitions; IEEE
    round-to-nearest-even to fp32 / fp16 / bf16.
``forms``
    Independent second forms used only to pin the direct loops: the
    per-channel im2col GEMV (Flash-DWC §2.1, Fig. 1), the tiled form with
    partial sums carried across tiles ("Tiles, halos and partial sums"), the
    gather form of dgrad, and the literal 180-degree-rotation form of the
    stride-1 dgrad (Flash-DWC §5.1).
``pages``
    The arithmetic the pages print: halo extents, storage budgets, the GEMM
    traffic model, and the Flash-DWC tile-model closed forms.

Every function here is pinned by ``tests/test_oracle_pins.py`` (the int64
loops, the page arithmetic, the fused and FP8 helpers) and
``tests/test_oracle_float_pins.py`` (the float64 loops and the magnitude
``mag``) against values the pages print, closed forms, special cases, brute
force and PyTorch's float64 convolution gradients; none is left "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dwconv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no -march flags, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            L, I, P = ctypes.c_long, ctypes.c_int, ctypes.c_void_p
            for name in ("dwo_fwd_f64", "dwo_fwd_i64"):
                fn = getattr(lib, name)
                fn.argtypes = [L] * 12 + [P, P, P, P, P, I]
                fn.restype = I
            for name in ("dwo_dgrad_f64", "dwo_dgrad_i64", "dwo_wgrad_f64", "dwo_wgrad_i64"):
                fn = getattr(lib, name)
                fn.argtypes = [L] * 12 + [P, P, P, P, I]
                fn.restype = I
            lib.dwo_out_extent.argtypes = [L] * 5
            lib.dwo_out_extent.restype = L
            _lib = lib
    return _lib


def default_threads() -> int:
    """Host threads the oracle uses: the cores this process may run on."""
    return len(os.sched_getaffinity(0))


def out_extent(X: int, F: int, S: int, D: int, P: int) -> int:
    """floor((X + 2P - D(F-1) - 1)/S) + 1, the floor convention of the oracle."""
    return int(_load().dwo_out_extent(X, F, S, D, P))


def _pair(v, what):
    """An int (both axes) or an (h, w) pair -> (h, w)."""
    if isinstance(v, (tuple, list)):
        if len(v) != 2:
            raise ValueError(f"{what} must be an int or an (h, w) pair")
        return int(v[0]), int(v[1])
    return int(v), int(v)


def _axes(stride, dilation, pad):
    (sh, sw), (dh, dw), (ph, pw) = _pair(stride, "stride"), _pair(dilation, "dilation"), _pair(pad, "pad")
    return sh, sw, dh, dw, ph, pw


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(a, integer):
    dt = np.int64 if integer else np.float64
    return np.ascontiguousarray(a, dtype=dt)


def _is_integer(*arrays) -> bool:
    kinds = {np.asarray(a).dtype.kind for a in arrays if a is not None}
    if kinds <= {"i", "u"}:
        return True
    if kinds & {"i", "u"}:
        raise TypeError("mixing integer and floating-point operands")
    return False


def fwd(x, w, bias=None, stride=1, dilation=1, pad=0, nthreads=None):
    """Forward DWC.  x [N,H,W,C], w [FH,FW,C], bias [C] or None; stride,
    dilation and pad each an int (both axes) or an (h, w) pair.

    Returns (y [N,OH,OW,C], mag [N,OH,OW,C]) in float64 or int64.
    """
    integer = _is_integer(x, w, bias)
    x, w = _prep(x, integer), _prep(w, integer)
    b = None if bias is None else _prep(bias, integer)
    N, H, W, C = x.shape
    FH, FW, Cw = w.shape
    if Cw != C or (b is not None and b.shape != (C,)):
        raise ValueError("channel mismatch")
    sh, sw, dh, dw, ph, pw = _axes(stride, dilation, pad)
    OH, OW = out_extent(H, FH, sh, dh, ph), out_extent(W, FW, sw, dw, pw)
    if OH <= 0 or OW <= 0:
        raise ValueError("empty output")
    y = np.empty((N, OH, OW, C), dtype=x.dtype)
    mag = np.empty_like(y)
    fn = _load().dwo_fwd_i64 if integer else _load().dwo_fwd_f64
    rc = fn(N, H, W, C, FH, FW, sh, sw, dh, dw, ph, pw, _ptr(x), _ptr(w), _ptr(b), _ptr(y),
            _ptr(mag), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle fwd rejected the arguments (code {rc})")
    return y, mag


def dgrad(dy, w, H, W, stride=1, dilation=1, pad=0, nthreads=None):
    """Input gradient (adjoint scatter).  dy [N,OH,OW,C] -> (dx [N,H,W,C], mag).
    stride, dilation, pad: int or (h, w) pair."""
    integer = _is_integer(dy, w)
    dy, w = _prep(dy, integer), _prep(w, integer)
    N, OH, OW, C = dy.shape
    FH, FW, Cw = w.shape
    if Cw != C:
        raise ValueError("channel mismatch")
    sh, sw, dh, dw, ph, pw = _axes(stride, dilation, pad)
    if (out_extent(H, FH, sh, dh, ph), out_extent(W, FW, sw, dw, pw)) != (OH, OW):
        raise ValueError("dy shape does not match the forward output of an H x W input")
    dx = np.empty((N, H, W, C), dtype=dy.dtype)
    mag = np.empty_like(dx)
    fn = _load().dwo_dgrad_i64 if integer else _load().dwo_dgrad_f64
    rc = fn(N, H, W, C, FH, FW, sh, sw, dh, dw, ph, pw, _ptr(dy), _ptr(w), _ptr(dx), _ptr(mag),
            nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle dgrad rejected the arguments (code {rc})")
    return dx, mag


def wgrad(x, dy, FH, FW, stride=1, dilation=1, pad=0, nthreads=None):
    """Weight gradient.  x [N,H,W,C], dy [N,OH,OW,C] -> (dw [FH,FW,C], mag).
    stride, dilation, pad: int or (h, w) pair."""
    integer = _is_integer(x, dy)
    x, dy = _prep(x, integer), _prep(dy, integer)
    N, H, W, C = x.shape
    sh, sw, dh, dw_, ph, pw = _axes(stride, dilation, pad)
    if (out_extent(H, FH, sh, dh, ph), out_extent(W, FW, sw, dw_, pw)) != dy.shape[1:3]:
        raise ValueError("dy shape does not match the forward output")
    if dy.shape[0] != N or dy.shape[3] != C:
        raise ValueError("batch/channel mismatch")
    dw = np.empty((FH, FW, C), dtype=x.dtype)
    mag = np.empty_like(dw)
    fn = _load().dwo_wgrad_i64 if integer else _load().dwo_wgrad_f64
    rc = fn(N, H, W, C, FH, FW, sh, sw, dh, dw_, ph, pw, _ptr(x), _ptr(dy), _ptr(dw), _ptr(mag),
            nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle wgrad rejected the arguments (code {rc})")
    return dw, mag


ACTIVATIONS = ("none", "relu", "relu6", "silu", "gelu")


def activation(v, act):
    """float64 activation functions, from their definitions: ReLU max(v, 0),
    ReLU6 min(max(v, 0), 6), SiLU v * sigmoid(v) = v / (1 + e^-v),
    GELU v * Phi(v) = v/2 * (1 + erf(v / sqrt(2)))."""
    import math
    v = np.asarray(v, dtype=np.float64)
    if act == "none":
        return v.copy()
    if act == "relu":
        return np.maximum(v, 0.0)
    if act == "relu6":
        return np.minimum(np.maximum(v, 0.0), 6.0)
    if act == "silu":
        return v / (1.0 + np.exp(-v))
    if act == "gelu":
        return 0.5 * v * (1.0 + np.vectorize(math.erf)(v / math.sqrt(2.0)))
    raise ValueError(f"unknown activation {act!r}")


# Storage formats: significand bits p (hidden bit included) and the frexp
# exponent e_min of the smallest normal number (v = m 2^e, 0.5 <= m < 1).
FORMATS = {"fp32": (24, -125), "fp16": (11, -13), "bf16": (8, -125)}


def round_to(v, fmt):
    """Round float64 values to the nearest value of a storage format, ties to
    even (IEEE 754 round-to-nearest-even), subnormals included; overflow is
    not handled (values stay far below the formats' largest numbers).  The
    integer significand q = rint(v 2^(p - e)) has p bits for a normal v."""
    p, emin = FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    e = np.maximum(e, emin)
    return np.ldexp(np.rint(np.ldexp(v, p - e)), e - p)


def affine_act(v, scale, shift, act, axis_len):
    """act(scale[c] v + shift[c]) over the last (channel) axis, float64;
    scale None = 1, shift None = 0."""
    s = np.ones(axis_len) if scale is None else np.asarray(scale, dtype=np.float64)
    t = np.zeros(axis_len) if shift is None else np.asarray(shift, dtype=np.float64)
    return activation(s * np.asarray(v, dtype=np.float64) + t, act)


def prologue(x, pre, fmt):
    """The fused layer's input x' = round_fmt(act(scale[c] x + shift[c])) for
    pre = (scale, shift, act), as the unfused BN+Act layer would store it in
    the storage format fmt (None: no rounding).  The padding of the
    convolution is applied to x', so padded positions stay zero."""
    x = np.asarray(x, dtype=np.float64)
    if pre is None:
        return x
    xa = affine_act(x, pre[0], pre[1], pre[2], x.shape[-1])
    return xa if fmt is None else round_to(xa, fmt)


def fwd_fused(x, w, bias=None, pre=None, post=None, fmt=None, stride=1, dilation=1, pad=0, nthreads=None):
    """Forward pass fused with a BN+Act before it and an affine map plus
    activation after it (Flash-DWC §5.2 "Kernel fusion": the BN+Act+DWC
    pattern, BN in inference form folded into a per-channel scale and shift):

        x' = round_fmt(act_pre(s_pre[c] x + t_pre[c]))            (pre)
        z  = DWC(x', w) + bias[c]                                 (zero padding of x')
        y  = act_post(s_post[c] z + t_post[c])                    (post)

    pre / post = (scale, shift, act) or None; float64 throughout except the
    rounding of x' to the storage format fmt.  Returns (y, mag) with mag =
    |s_post| mag_conv + |t_post|, the magnitude of act_post's argument
    (mag_conv = sum |w x'| + |bias|)."""
    xq = prologue(x, pre, fmt)
    z, mag = fwd(xq, np.asarray(w, dtype=np.float64), None if bias is None else np.asarray(bias, dtype=np.float64),
                 stride, dilation, pad, nthreads)
    if post is None:
        return z, mag
    C = z.shape[-1]
    s = np.ones(C) if post[0] is None else np.asarray(post[0], dtype=np.float64)
    t = np.zeros(C) if post[1] is None else np.asarray(post[1], dtype=np.float64)
    return activation(s * z + t, post[2]), np.abs(s) * mag + np.abs(t)


def decode_e4m3(bits):
    """Values of FP8 E4M3 codes (uint8), float64, from the format's definition
    (OCP 8-bit floating point, E4M3): sign bit, 4 exponent bits with bias 7,
    3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; the code
    S.1111.111 is NaN and there are no infinities (largest value 448)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def dbias(dy):
    """Bias gradient.  dy [N,OH,OW,C] -> (db [C], mag [C]).

    The forward pass adds bias[c] once to every output of channel c
    ("Tiles, halos and partial sums"), so the adjoint of the bias term is
    the plain sum of dy over n, oh and ow: db[c] = sum dy[n,oh,ow,c];
    mag[c] = sum |dy[n,oh,ow,c]|.  float64 or int64.
    """
    integer = _is_integer(dy)
    dy = _prep(dy, integer)
    if dy.ndim != 4:
        raise ValueError("dy must be [N,OH,OW,C]")
    flat = dy.reshape(-1, dy.shape[3])
    return flat.sum(axis=0), np.abs(flat).sum(axis=0)


from . import forms, pages  # noqa: E402  (pure-Python helpers, no C needed)

__all__ = ["build", "fwd", "fwd_fused", "decode_e4m3", "prologue", "affine_act", "activation", "ACTIVATIONS", "round_to", "FORMATS", "dgrad", "wgrad", "dbias", "out_extent",
           "default_threads", "forms", "pages"]
