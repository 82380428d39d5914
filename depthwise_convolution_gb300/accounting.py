"""Algorithmic work of each pass, for throughput and roofline reporting.

Flops: "nominal" = 2 * N * OH * OW * C * FH * FW (the Flash-DWC convention,
§2.2 and §6.1, counting padding taps); "valid" = 2 * (taps that land inside
the input).  Bytes: unique tensor bytes, each element counted once -- the
lower bound "Tiles, halos and partial sums" distinguishes from the tile
transfers a kernel actually makes:
  fwd    read the input elements some tap touches + w + bias, write y
  dgrad  read dy + w, write all of dx
  wgrad  read the touched input elements + dy, write dw (fp32)
"""
from __future__ import annotations

ELEM = {"int8": 1, "fp32": 4, "fp16": 2, "bf16": 2, "fp8": 1}


def out_extent(X, F, S, D, P):
    return (X + 2 * P - D * (F - 1) - 1) // S + 1


def _axis_valid_taps(X, F, S, D, P):
    O = out_extent(X, F, S, D, P)
    return sum(1 for o in range(O) for f in range(F) if 0 <= o * S - P + f * D < X)


def _axis_touched(X, F, S, D, P):
    O = out_extent(X, F, S, D, P)
    return len({o * S - P + f * D for o in range(O) for f in range(F)} & set(range(X)))


def nominal_flops(N, H, W, C, FH, FW, S, D, P):
    return 2 * N * out_extent(H, FH, S, D, P) * out_extent(W, FW, S, D, P) * C * FH * FW


def valid_flops(N, H, W, C, FH, FW, S, D, P):
    return 2 * N * C * _axis_valid_taps(H, FH, S, D, P) * _axis_valid_taps(W, FW, S, D, P)


def unique_bytes(pass_name, dtype, N, H, W, C, FH, FW, S, D, P, bias=False):
    e = ELEM[dtype]
    OH, OW = out_extent(H, FH, S, D, P), out_extent(W, FW, S, D, P)
    touched = N * _axis_touched(H, FH, S, D, P) * _axis_touched(W, FW, S, D, P) * C
    w = FH * FW * C * e
    if pass_name == "fwd":
        ybytes = N * OH * OW * C * (4 if dtype == "int8" else 2 if dtype == "fp8" else e)  # int32 / bf16 y
        return touched * e + w + (C * 4 if bias else 0) + ybytes
    if pass_name == "dgrad":
        return N * OH * OW * C * e + w + N * H * W * C * e
    if pass_name == "wgrad":
        return touched * e + N * OH * OW * C * e + FH * FW * C * 4
    raise ValueError(pass_name)
