"""Shared helpers for the GPU parity tests: run a pass through the library,
run the oracle on the same quantised inputs, compare element by element.

Tolerances (per output element, mag = sum |products| (+ |bias|) from the oracle):
  int8 -> int32          bit-exact (int64 oracle reduced mod 2^32)
  fp32                   |gpu - ref| <= 1e-5 * mag
  fp16 / bf16 inputs     |gpu - ref| <= 2e-3 * mag, plus, for 16-bit outputs,
                         half a unit in the last place of the output format at
                         max(|ref|, |gpu|): the rounding the output type itself
                         forces, which an fp32-accumulation bound cannot cover
                         (bf16 keeps 8 significant bits, so rounding alone can
                         reach 2^-8 |y|).  wgrad writes fp32 and gets no such term.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from depthwise_convolution_gb300 import ops

TOL = {"fp32": 1e-5, "fp16": 2e-3, "bf16": 2e-3, "fp8": 2e-3}
SIG_BITS = {"fp16": 11, "bf16": 8}      # significand bits including the hidden one
MIN_EXP = {"fp16": -14, "bf16": -126}   # exponent of the smallest normal number
TORCH = {"int8": torch.int8, "fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16,
         "fp8": getattr(torch, "float8_e4m3fn", None)}
OUT16 = {"fp16": "fp16", "bf16": "bf16", "fp8": "bf16"}  # 16-bit output format per input dtype
GUARD = 256                              # guard elements on each side of an output


def half_ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    p = SIG_BITS[dtype]
    _, e = np.frexp(np.abs(v))           # |v| = m * 2^e, m in [0.5, 1)
    e = np.maximum(e - 1, MIN_EXP[dtype])  # unbiased exponent, subnormals share the minimum
    return np.ldexp(1.0, e - p)          # half of 2^(e - p + 1)


def to64(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype in (torch.int8, torch.int32):
        return t.to(torch.int64).numpy()
    if TORCH["fp8"] is not None and t.dtype == TORCH["fp8"]:
        return oracle.decode_e4m3(t.view(torch.uint8).numpy())  # from the format's bits
    return t.to(torch.float64).numpy()


def compare(got: np.ndarray, ref: np.ndarray, mag: np.ndarray, dtype: str, out16: bool, what: str):
    """Assert the tolerance; return the largest err / mag seen."""
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if dtype == "int8":
        expect = ((ref + 2**31) % 2**32) - 2**31
        bad = np.nonzero(got != expect)
        assert bad[0].size == 0, f"{what}: {bad[0].size} int32 mismatches, first at {tuple(b[0] for b in bad)}"
        return 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = TOL[dtype] * mag
    if out16:
        bound = bound + half_ulp(np.maximum(np.abs(ref), np.abs(got)), OUT16[dtype])
    over = err > bound
    if over.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(over.sum())} elements over tolerance; worst at {i}: "
                             f"gpu={got[i]!r} ref={ref[i]!r} mag={mag[i]!r} bound={bound[i]!r}")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(mag > 0, err / mag, 0.0)
    return float(ratio.max()) if ratio.size else 0.0


class Guarded:
    """An output tensor inside a larger buffer whose ends hold a bit pattern
    that must survive the call (an out-of-bounds write shows up there)."""

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape))
        self.buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
        raw = self.buf.view(torch.uint8)
        raw.fill_(0xA5)
        self.guard_bytes = GUARD * self.buf.element_size()
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        self.t.fill_(float("nan") if dtype.is_floating_point else -12345)

    def check(self, what):
        raw = self.buf.view(torch.uint8)
        head = raw[:self.guard_bytes].cpu()
        tail = raw[-self.guard_bytes:].cpu()
        assert bool((head == 0xA5).all()) and bool((tail == 0xA5).all()), f"{what}: guard band overwritten"


def _pair(v):
    return (int(v[0]), int(v[1])) if isinstance(v, (tuple, list)) else (int(v), int(v))


def out_hw(H, W, FH, FW, S, D, P):
    """Forward output size; S, D, P each an int or an (h, w) pair."""
    (sh, sw), (dh, dw), (ph, pw) = _pair(S), _pair(D), _pair(P)
    return oracle.out_extent(H, FH, sh, dh, ph), oracle.out_extent(W, FW, sw, dw, pw)


def random_inputs(dtype, N, H, W, C, FH, FW, S, D, P, seed, bias=True):
    from depthwise_convolution_gb300 import synthetic as syn
    wl = syn.Workload("case", dtype, N, H, W, C, FH, FW, S, D, P, bias, ("fwd", "dgrad", "wgrad"), seed)
    OH, OW = out_hw(H, W, FH, FW, S, D, P)
    if dtype == "int8":
        d = syn.make_inputs(wl)
        d["dy"] = None
    else:
        d = syn.make_inputs(wl, dy_hw=(OH, OW))
    return d


def check_fwd(d, dtype, S, D, P, images=None, what="fwd"):
    x, w, b = d["x"], d["w"], d["bias"]
    N, H, W, C = x.shape
    FH, FW = w.shape[:2]
    OH, OW = out_hw(H, W, FH, FW, S, D, P)
    out_dtype = torch.int32 if dtype == "int8" else torch.bfloat16 if dtype == "fp8" else TORCH[dtype]
    g = Guarded((N, OH, OW, C), out_dtype)
    y = ops.dwconv_fwd(x.cuda(), w.cuda(), None if b is None else b.cuda(), S, D, P, out=g.t)
    ops.dwconv_check_device_errors()
    g.check(what)
    imgs = list(range(N)) if images is None else sorted(set(i % N for i in images))
    ref, mag = oracle.fwd(to64(x)[imgs], to64(w), None if b is None else to64(b), S, D, P)
    return compare(to64(y[imgs]), ref, mag, dtype, dtype in ("fp16", "bf16", "fp8"), what)


def check_dgrad(d, dtype, S, D, P, images=None, what="dgrad"):
    dy, w = d["dy"], d["w"]
    N, H, W, C = d["x"].shape
    g = Guarded((N, H, W, C), TORCH[dtype])
    dx = ops.dwconv_bwd_data(dy.cuda(), w.cuda(), H, W, S, D, P, out=g.t)
    ops.dwconv_check_device_errors()
    g.check(what)
    imgs = list(range(N)) if images is None else sorted(set(i % N for i in images))
    ref, mag = oracle.dgrad(to64(dy[imgs]), to64(w), H, W, S, D, P)
    return compare(to64(dx[imgs]), ref, mag, dtype, dtype in ("fp16", "bf16"), what)


def check_dbias(d, dtype, what="dbias"):
    dy = d["dy"]
    C = dy.shape[3]
    g = Guarded((C,), torch.float32)
    db = ops.dwconv_bwd_bias(dy.cuda(), out=g.t)
    ops.dwconv_check_device_errors()
    g.check(what)
    ref, mag = oracle.dbias(to64(dy))
    return compare(to64(db), ref, mag, dtype, False, what)


def check_wgrad(d, dtype, S, D, P, what="wgrad"):
    x, dy = d["x"], d["dy"]
    FH, FW, C = d["w"].shape
    g = Guarded((FH, FW, C), torch.float32)
    dw = ops.dwconv_bwd_filter(x.cuda(), dy.cuda(), FH, FW, S, D, P, out=g.t)
    ops.dwconv_check_device_errors()
    g.check(what)
    ref, mag = oracle.wgrad(to64(x), to64(dy), FH, FW, S, D, P)
    return compare(to64(dw), ref, mag, dtype, False, what)


# Largest slope of each activation (|act'| <= LIP): an error e in the
# activation's argument moves its value by at most LIP * e.  SiLU' peaks at
# 1.0998 (v = 2.40), GELU' at 1.1289 (v = 1.41).
LIP = {"none": 1.0, "relu": 1.0, "relu6": 1.0, "silu": 1.1, "gelu": 1.13}


def check_fused(d, dtype, S, D, P, pre=None, post=None, images=None, what="fused"):
    """Fused forward pass against oracle.fwd_fused.  pre / post: (scale,
    shift, act) with CPU float32 scale / shift (or None).

    Tolerance: LIP[act_post] * (TOL * mag + |s_post| * E_pre) + 1e-6 * mag,
    plus half an ulp of 16-bit outputs, where mag is the oracle's magnitude
    of act_post's argument and E_pre = sum |w| * ulp(x') bounds a one-ulp
    difference in the rounding of any prologue value x' to the storage type
    (the kernel evaluates the prologue in fp32, the oracle in float64, so a
    value within a few fp32 ulps of a rounding boundary may round either way).
    """
    x, w, b = d["x"], d["w"], d["bias"]
    N, H, W, C = x.shape
    FH, FW = w.shape[:2]
    OH, OW = out_hw(H, W, FH, FW, S, D, P)
    cuda = lambda v: None if v is None else v.cuda()
    kw = {}
    if pre is not None:
        kw.update(in_scale=cuda(pre[0]), in_shift=cuda(pre[1]), in_act=pre[2])
    if post is not None:
        kw.update(out_scale=cuda(post[0]), out_shift=cuda(post[1]), out_act=post[2])
    g = Guarded((N, OH, OW, C), torch.bfloat16 if dtype == "fp8" else TORCH[dtype])
    y = ops.dwconv_fwd_fused(x.cuda(), w.cuda(), cuda(b), stride=S, dilation=D, pad=P, out=g.t, **kw)
    ops.dwconv_check_device_errors()
    g.check(what)
    kernel = ops.dwconv_last_kernel()
    imgs = list(range(N)) if images is None else sorted(set(i % N for i in images))
    f64 = lambda v: None if v is None else to64(v)
    opre = None if pre is None else (f64(pre[0]), f64(pre[1]), pre[2])
    opost = None if post is None else (f64(post[0]), f64(post[1]), post[2])
    fmt = dtype if dtype in ("fp16", "bf16", "fp32") else None
    ref, mag = oracle.fwd_fused(to64(x)[imgs], to64(w), f64(b), pre=opre, post=opost, fmt=fmt,
                                stride=S, dilation=D, pad=P)
    got = to64(y[imgs])
    lip = LIP[post[2]] if post is not None else 1.0
    s_post = np.ones(C) if post is None or post[0] is None else np.abs(f64(post[0]))
    e_pre = 0.0
    if pre is not None and dtype in ("fp16", "bf16"):
        xq = oracle.prologue(to64(x)[imgs], opre, fmt)
        e_pre, _ = oracle.fwd(2 * half_ulp(xq, dtype), np.abs(to64(w)), None, S, D, P)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = lip * (TOL[dtype] * mag + s_post * e_pre) + 1e-6 * mag
    if dtype in OUT16:
        bound = bound + half_ulp(np.maximum(np.abs(ref), np.abs(got)), OUT16[dtype])
    over = err > bound
    if over.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what} [{kernel}]: {int(over.sum())} elements over tolerance; worst at {i}: "
                             f"gpu={got[i]!r} ref={ref[i]!r} mag={mag[i]!r} bound={bound[i]!r}")
    return kernel
