"""Second, independent forms of the operator, used only to pin the direct loops.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Small inputs only:
these are written for clarity, with Python loops over tiles and taps.
"""
from __future__ import annotations

import numpy as np

from . import pages


def _out(X, F, S, D, P):
    return (X + 2 * P - D * (F - 1) - 1) // S + 1


def im2col_gemv_fwd(x, w, bias=None, stride=1, dilation=1, pad=0):
    """Flash-DWC §2.1 and Fig. 1: per channel, the im2col matrix of every
    output position (rows) by every filter tap (columns, zero where the tap
    falls in the padding) times the flattened filter vector, plus bias."""
    x = np.asarray(x)
    w = np.asarray(w)
    N, H, W, C = x.shape
    FH, FW, _ = w.shape
    S, D, P = stride, dilation, pad
    OH, OW = _out(H, FH, S, D, P), _out(W, FW, S, D, P)
    dt = np.int64 if x.dtype.kind in "iu" else np.float64
    y = np.zeros((N, OH, OW, C), dtype=dt)
    for c in range(C):
        A = np.zeros((N * OH * OW, FH * FW), dtype=dt)
        row = 0
        for n in range(N):
            for oh in range(OH):
                for ow in range(OW):
                    for fh in range(FH):
                        for fw in range(FW):
                            ih, iw = oh * S - P + fh * D, ow * S - P + fw * D
                            if 0 <= ih < H and 0 <= iw < W:
                                A[row, fh * FW + fw] = x[n, ih, iw, c]
                    row += 1
        v = w[:, :, c].reshape(FH * FW).astype(dt)
        col = A @ v
        if bias is not None:
            col = col + dt(np.asarray(bias)[c])
        y[..., c] = col.reshape(N, OH, OW)
    return y


def tiled_fwd(x, w, bias=None, stride=1, dilation=1, pad=0, Th=2, Tw=2, Tc=2,
              row_groups=2, bias_mode="once"):
    """The forward pass computed tile by tile ("Tiles, halos and partial sums").

    Output tiles of Th x Tw positions and Tc channels (tails masked).  Each tile
    stages its input halo of halo_extent(Th) x halo_extent(Tw) positions, with
    the padding generated as zeros rather than read.  The FH filter rows are
    split into ``row_groups`` groups (the 1-D decomposition of Flash-DWC §3.3);
    each group adds its partial sum to the same full-precision accumulator and
    the bias enters once, with the first group.

    ``bias_mode="every_group"`` is a deliberately wrong variant used only by a
    test to show that a bias added more than once is caught.
    """
    x = np.asarray(x)
    w = np.asarray(w)
    N, H, W, C = x.shape
    FH, FW, _ = w.shape
    S, D, P = stride, dilation, pad
    OH, OW = _out(H, FH, S, D, P), _out(W, FW, S, D, P)
    dt = np.int64 if x.dtype.kind in "iu" else np.float64
    xb = x.astype(dt)
    wb = w.astype(dt)
    bb = None if bias is None else np.asarray(bias).astype(dt)
    hh, hw = pages.halo_extent(Th, S, FH, D), pages.halo_extent(Tw, S, FW, D)
    bounds = np.linspace(0, FH, row_groups + 1).astype(int)
    y = np.zeros((N, OH, OW, C), dtype=dt)
    for c0 in range(0, C, Tc):
        cv = min(Tc, C - c0)                       # valid channels in this tile
        for n in range(N):
            for oh0 in range(0, OH, Th):
                for ow0 in range(0, OW, Tw):
                    ih0, iw0 = oh0 * S - P, ow0 * S - P
                    halo = np.zeros((hh, hw, Tc), dtype=dt)   # padding generated
                    for a in range(hh):
                        for b in range(hw):
                            ih, iw = ih0 + a, iw0 + b
                            if 0 <= ih < H and 0 <= iw < W:
                                halo[a, b, :cv] = xb[n, ih, iw, c0:c0 + cv]
                    wt = np.zeros((FH, FW, Tc), dtype=dt)
                    wt[:, :, :cv] = wb[:, :, c0:c0 + cv]
                    acc = np.zeros((Th, Tw, Tc), dtype=dt)
                    for g in range(row_groups):
                        if bb is not None and (g == 0 or bias_mode == "every_group"):
                            acc[:, :, :cv] += bb[c0:c0 + cv]
                        for fh in range(bounds[g], bounds[g + 1]):
                            for fw in range(FW):
                                for t in range(Th):
                                    for u in range(Tw):
                                        acc[t, u] += wt[fh, fw] * halo[t * S + fh * D, u * S + fw * D]
                    th_v, tw_v = min(Th, OH - oh0), min(Tw, OW - ow0)
                    y[n, oh0:oh0 + th_v, ow0:ow0 + tw_v, c0:c0 + cv] = acc[:th_v, :tw_v, :cv]
    return y


def dgrad_gather(dy, w, H, W, stride=1, dilation=1, pad=0):
    """dgrad written per input element: the sum over taps (fh, fw) whose output
    position oh = (ih + P - fh*D)/S is a whole number inside [0, OH)."""
    dy = np.asarray(dy)
    w = np.asarray(w)
    N, OH, OW, C = dy.shape
    FH, FW, _ = w.shape
    S, D, P = stride, dilation, pad
    dt = np.int64 if dy.dtype.kind in "iu" else np.float64
    dx = np.zeros((N, H, W, C), dtype=dt)
    for ih in range(H):
        for iw in range(W):
            acc = np.zeros((N, C), dtype=dt)
            for fh in range(FH):
                th = ih + P - fh * D
                if th % S != 0 or not (0 <= th // S < OH):
                    continue
                for fw in range(FW):
                    tw = iw + P - fw * D
                    if tw % S != 0 or not (0 <= tw // S < OW):
                        continue
                    acc += w[fh, fw].astype(dt) * dy[:, th // S, tw // S, :].astype(dt)
            dx[:, ih, iw, :] = acc
    return dx


def dgrad_rot180_stride1(dy, w, H, W, dilation=1, pad=0):
    """Flash-DWC §5.1: for stride 1, dgrad is the forward pass over dy with the
    filter rotated by 180 degrees and padding D(FH-1)-P (here via the direct
    loop of the oracle; requires 0 <= P <= D(FH-1) and the same along width)."""
    from . import fwd
    FH, FW, _ = np.asarray(w).shape
    D = dilation
    ph, pw = D * (FH - 1) - pad, D * (FW - 1) - pad
    if ph < 0 or pw < 0 or ph != pw:
        raise ValueError("this form needs 0 <= P <= D(FH-1) and square padding")
    wr = np.ascontiguousarray(np.asarray(w)[::-1, ::-1, :])
    dx, _ = fwd(dy, wr, None, stride=1, dilation=D, pad=ph)
    assert dx.shape[1:3] == (H, W)
    return dx


def conv1d_zero_pad(v, f):
    """"Outline of Programming Massively Parallel Processors", Convolution /
    Introduction: each output is the weighted sum of the 2r+1 inputs centred on
    it, with positions past either end read as zero."""
    v = list(v)
    r = (len(f) - 1) // 2
    out = []
    for i in range(len(v)):
        s = 0
        for j in range(len(f)):
            k = i - r + j
            if 0 <= k < len(v):
                s += f[j] * v[k]
        out.append(s)
    return out


def touched_input_positions(H, W, FH, FW, stride=1, dilation=1, pad=0):
    """Brute force: the set of input (ih, iw) positions any valid tap reads."""
    OH, OW = _out(H, FH, stride, dilation, pad), _out(W, FW, stride, dilation, pad)
    rows = {oh * stride - pad + fh * dilation for oh in range(OH) for fh in range(FH)}
    cols = {ow * stride - pad + fw * dilation for ow in range(OW) for fw in range(FW)}
    rows = {r for r in rows if 0 <= r < H}
    cols = {c for c in cols if 0 <= c < W}
    return rows, cols


def valid_tap_count(H, W, FH, FW, stride=1, dilation=1, pad=0):
    """Brute force: number of (oh, ow, fh, fw) whose tap lands inside the input."""
    OH, OW = _out(H, FH, stride, dilation, pad), _out(W, FW, stride, dilation, pad)
    rows = sum(1 for oh in range(OH) for fh in range(FH) if 0 <= oh * stride - pad + fh * dilation < H)
    cols = sum(1 for ow in range(OW) for fw in range(FW) if 0 <= ow * stride - pad + fw * dilation < W)
    return rows * cols
