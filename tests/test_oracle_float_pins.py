"""Pins for the oracle's float64 passes and for its per-element magnitude.

The floating-point parity tests compare the CUDA path with the float64 copies
of the oracle's loops (``fwd``, ``dgrad``, ``wgrad`` on float data) and scale
their bound by the ``mag`` those loops return, so both are pinned here, each
against something other than the oracle itself:

* the adjoint identity of the bias-free forward map (a textbook property of
  the definition in Flash-DWC §2.1 and of the training passes of §5.1), the
  gather form of dgrad, and the stride-1 "rotate the filter by 180 degrees"
  form of §5.1, all run through the float64 code on integer-valued data, where
  float64 arithmetic is exact, so they hold with equality;
* PyTorch's float64 ``conv2d(groups=C)`` and its autograd gradients on random
  normal data (a library routine with the same definition, test-only);
* ``mag`` = |bias| + sum |product|: it is exactly the value of the same pass
  on the absolute values of its operands, since |a*b| = |a|*|b| holds exactly
  in IEEE arithmetic and the loops add in the same order.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle import forms

rng = np.random.default_rng(777)


def fint(shape, lo=-9, hi=9):
    """Integer-valued float64 data: every sum the small cases form is exact."""
    return rng.integers(lo, hi, size=shape, endpoint=True).astype(np.float64)


def cases():
    """(N,H,W,C,FH,FW,S,D,P): every stride / dilation / padding combination
    with a non-empty output, asymmetric filters included."""
    out = []
    for S, D in itertools.product((1, 2, 3), (1, 2)):
        for FH, FW in ((1, 1), (3, 3), (2, 3), (3, 1), (5, 4)):
            for P in range(0, D * (max(FH, FW) - 1) + 2):
                H, W = 7, 6
                if oracle.out_extent(H, FH, S, D, P) >= 1 and oracle.out_extent(W, FW, S, D, P) >= 1:
                    out.append((2, H, W, 3, FH, FW, S, D, P))
    return out


CASES = cases()


def torch_dwconv(x, w, b, S, D, P):
    """NHWC float64 arrays -> torch tensors in NCHW / [C,1,FH,FW] with grad."""
    xt = torch.from_numpy(x).permute(0, 3, 1, 2).contiguous().requires_grad_(True)
    wt = torch.from_numpy(w).permute(2, 0, 1).unsqueeze(1).contiguous().requires_grad_(True)
    bt = None if b is None else torch.from_numpy(b)
    yt = torch.nn.functional.conv2d(xt, wt, bt, stride=S, padding=P, dilation=D, groups=x.shape[3])
    return xt, wt, yt


# ------------------------------------------------- float64 dgrad and wgrad

@pytest.mark.parametrize("case", CASES)
def test_f64_adjoint_identity_exact(case):
    """<fwd0(x,w), dy> = <x, dgrad(dy,w)> = <w, wgrad(x,dy)> through the
    float64 loops; integer-valued data keeps every sum exact."""
    N, H, W, C, FH, FW, S, D, P = case
    x, w = fint((N, H, W, C)), fint((FH, FW, C))
    y, _ = oracle.fwd(x, w, None, S, D, P)
    assert y.dtype == np.float64
    dy = fint(y.shape)
    dx, _ = oracle.dgrad(dy, w, H, W, S, D, P)
    dw, _ = oracle.wgrad(x, dy, FH, FW, S, D, P)
    assert dx.dtype == np.float64 and dw.dtype == np.float64
    lhs = float(np.sum(y * dy))
    assert lhs == float(np.sum(x * dx))
    assert lhs == float(np.sum(w * dw))


@pytest.mark.parametrize("case", CASES)
def test_f64_adjoint_identity_per_element(case):
    """The adjoint identity for each channel on its own (channels never mix in
    a depthwise convolution, so a channel index swapped anywhere fails it)."""
    N, H, W, C, FH, FW, S, D, P = case
    x, w = fint((N, H, W, C)), fint((FH, FW, C))
    y, _ = oracle.fwd(x, w, None, S, D, P)
    dy = fint(y.shape)
    dx, _ = oracle.dgrad(dy, w, H, W, S, D, P)
    dw, _ = oracle.wgrad(x, dy, FH, FW, S, D, P)
    for c in range(C):
        lhs = float(np.sum(y[..., c] * dy[..., c]))
        assert lhs == float(np.sum(x[..., c] * dx[..., c]))
        assert lhs == float(np.sum(w[..., c] * dw[..., c]))


@pytest.mark.parametrize("case", CASES[::2])
def test_f64_dgrad_gather_form_equals_scatter_form(case):
    N, H, W, C, FH, FW, S, D, P = case
    w = fint((FH, FW, C))
    dy = fint((N, oracle.out_extent(H, FH, S, D, P), oracle.out_extent(W, FW, S, D, P), C))
    dx, _ = oracle.dgrad(dy, w, H, W, S, D, P)
    assert np.array_equal(dx, forms.dgrad_gather(dy, w, H, W, S, D, P))


@pytest.mark.parametrize("F,D,P", [(3, 1, 1), (5, 1, 2), (3, 2, 2), (5, 2, 4), (7, 1, 3), (4, 1, 0), (2, 1, 1)])
def test_f64_stride1_dgrad_is_forward_with_rotated_filter(F, D, P):
    """Flash-DWC §5.1: for stride 1 the input gradient is the forward pass of
    dy with the 180-degree-rotated filter and padding D(F-1)-P."""
    H, W, C = 10, 9, 3
    w = fint((F, F, C))
    dy = fint((2, oracle.out_extent(H, F, 1, D, P), oracle.out_extent(W, F, 1, D, P), C))
    dx, _ = oracle.dgrad(dy, w, H, W, 1, D, P)
    assert np.array_equal(dx, forms.dgrad_rot180_stride1(dy, w, H, W, D, P))


@pytest.mark.parametrize("case", CASES[::3])
def test_f64_wgrad_is_the_correlation_of_x_with_dy(case):
    """dw[fh,fw,c] = sum over output sites of dy * x at the tapped input site:
    with dy one-hot at (n, oh, ow) the gradient is the tapped input window."""
    N, H, W, C, FH, FW, S, D, P = case
    x = fint((N, H, W, C))
    OH, OW = oracle.out_extent(H, FH, S, D, P), oracle.out_extent(W, FW, S, D, P)
    for (n, oh, ow) in ((0, 0, 0), (N - 1, OH - 1, OW - 1), (N - 1, OH // 2, 0)):
        dy = np.zeros((N, OH, OW, C))
        dy[n, oh, ow, :] = 1.0
        dw, _ = oracle.wgrad(x, dy, FH, FW, S, D, P)
        expect = np.zeros((FH, FW, C))
        for fh in range(FH):
            for fw in range(FW):
                ih, iw = oh * S - P + fh * D, ow * S - P + fw * D
                if 0 <= ih < H and 0 <= iw < W:
                    expect[fh, fw] = x[n, ih, iw]
        assert np.array_equal(dw, expect)


@pytest.mark.parametrize("case", CASES[::3])
def test_f64_gradients_match_torch_autograd(case):
    """Random normal float64 data: dgrad and wgrad equal PyTorch's autograd
    gradients of <conv2d(x, w, groups=C), dy>, to float64 rounding."""
    N, H, W, C, FH, FW, S, D, P = case
    x, w = rng.standard_normal((N, H, W, C)), rng.standard_normal((FH, FW, C))
    xt, wt, yt = torch_dwconv(x, w, None, S, D, P)
    dy = rng.standard_normal(tuple(yt.permute(0, 2, 3, 1).shape))
    gx, gw = torch.autograd.grad(yt, (xt, wt), torch.from_numpy(dy).permute(0, 3, 1, 2))
    dx, mdx = oracle.dgrad(dy, w, H, W, S, D, P)
    dw, mdw = oracle.wgrad(x, dy, FH, FW, S, D, P)
    gx = gx.permute(0, 2, 3, 1).numpy()
    gw = gw.squeeze(1).permute(1, 2, 0).numpy()
    # Each result is a sum of at most FH*FW (dgrad) or N*OH*OW (wgrad) products;
    # two summation orders differ by a few units of 2^-52 times the magnitude.
    assert np.all(np.abs(dx - gx) <= 1e-13 * (mdx + 1))
    assert np.all(np.abs(dw - gw) <= 1e-13 * (mdw + 1))


def test_f64_stride2_dilation2_odd_positions_get_no_gradient():
    H = W = 12
    w = rng.standard_normal((5, 5, 2))
    dy = rng.standard_normal((1, 6, 6, 2))
    dx, mag = oracle.dgrad(dy, w, H, W, 2, 2, 4)
    assert not dx[:, 1::2].any() and not dx[:, :, 1::2].any()
    assert not mag[:, 1::2].any() and not mag[:, :, 1::2].any()
    assert np.all(mag[:, ::2, ::2] > 0)


# --------------------------------------------------------------- magnitude

@pytest.mark.parametrize("case", CASES[::2])
def test_mag_is_the_pass_on_absolute_values(case):
    """mag of every pass equals, exactly, that pass applied to |operands|."""
    N, H, W, C, FH, FW, S, D, P = case
    x, w, b = rng.standard_normal((N, H, W, C)), rng.standard_normal((FH, FW, C)), rng.standard_normal(C)
    y, mag = oracle.fwd(x, w, b, S, D, P)
    assert np.array_equal(mag, oracle.fwd(np.abs(x), np.abs(w), np.abs(b), S, D, P)[0])
    y0, mag0 = oracle.fwd(x, w, None, S, D, P)
    assert np.array_equal(mag0, oracle.fwd(np.abs(x), np.abs(w), None, S, D, P)[0])
    dy = rng.standard_normal(y.shape)
    dx, mdx = oracle.dgrad(dy, w, H, W, S, D, P)
    assert np.array_equal(mdx, oracle.dgrad(np.abs(dy), np.abs(w), H, W, S, D, P)[0])
    dw, mdw = oracle.wgrad(x, dy, FH, FW, S, D, P)
    assert np.array_equal(mdw, oracle.wgrad(np.abs(x), np.abs(dy), FH, FW, S, D, P)[0])
    db, mdb = oracle.dbias(dy)
    assert np.array_equal(mdb, oracle.dbias(np.abs(dy))[0])


@pytest.mark.parametrize("case", CASES[1::4])
def test_mag_int64_is_the_pass_on_absolute_values(case):
    N, H, W, C, FH, FW, S, D, P = case
    ri = lambda s: rng.integers(-9, 9, size=s, endpoint=True)  # noqa: E731
    x, w, b = ri((N, H, W, C)), ri((FH, FW, C)), ri((C,))
    y, mag = oracle.fwd(x, w, b, S, D, P)
    assert np.array_equal(mag, oracle.fwd(np.abs(x), np.abs(w), np.abs(b), S, D, P)[0])
    dy = ri(y.shape)
    assert np.array_equal(oracle.dgrad(dy, w, H, W, S, D, P)[1],
                          oracle.dgrad(np.abs(dy), np.abs(w), H, W, S, D, P)[0])
    assert np.array_equal(oracle.wgrad(x, dy, FH, FW, S, D, P)[1],
                          oracle.wgrad(np.abs(x), np.abs(dy), FH, FW, S, D, P)[0])


def test_mag_closed_forms():
    """Hand-computed magnitudes: a 3x3 all-ones filter over an input of -2,
    bias -1.5, pad 1: interior 9*2 + 1.5, edge 6*2 + 1.5, corner 4*2 + 1.5;
    dgrad of dy = -1 through filter values -3: 9*3 inside, 4*3 in a corner;
    wgrad of x = -2 and dy = 0.5 on a 4x4 map: the centre tap sums 16 products
    of magnitude 1, a corner tap 9."""
    x = np.full((1, 4, 4, 1), -2.0)
    w = np.ones((3, 3, 1))
    y, mag = oracle.fwd(x, w, np.array([-1.5]), 1, 1, 1)
    assert mag[0, 1, 1, 0] == 19.5 and mag[0, 0, 1, 0] == 13.5 and mag[0, 0, 0, 0] == 9.5
    assert y[0, 1, 1, 0] == -19.5 and y[0, 0, 0, 0] == -9.5
    dx, mdx = oracle.dgrad(np.full((1, 4, 4, 1), -1.0), np.full((3, 3, 1), -3.0), 4, 4, 1, 1, 1)
    assert mdx[0, 1, 1, 0] == 27.0 and mdx[0, 0, 0, 0] == 12.0 and dx[0, 1, 1, 0] == 27.0
    dw, mdw = oracle.wgrad(x, np.full((1, 4, 4, 1), 0.5), 3, 3, 1, 1, 1)
    assert mdw[1, 1, 0] == 16.0 and mdw[0, 0, 0] == 9.0 and dw[1, 1, 0] == -16.0


def test_mag_bounds_the_value_and_cancellation_shows():
    """|value| <= mag always; with products of both signs the gap is visible
    (a mag that were computed as |value| would fail the strict check)."""
    x = np.array([1.0, -1.0, 2.0, -2.0]).reshape(1, 1, 4, 1)
    w = np.ones((1, 3, 1))
    y, mag = oracle.fwd(x, w, None, 1, 1, (0, 1))
    assert y[0, 0, :, 0].tolist() == [0.0, 2.0, -1.0, 0.0]
    assert mag[0, 0, :, 0].tolist() == [2.0, 4.0, 5.0, 4.0]
    xs, ws = rng.standard_normal((2, 9, 8, 4)), rng.standard_normal((3, 3, 4))
    ys, ms = oracle.fwd(xs, ws, None, 1, 1, 1)
    assert np.all(np.abs(ys) <= ms) and np.any(np.abs(ys) < ms)


def test_fused_mag_is_the_affine_of_the_convolution_mag():
    """Fused forward with a post affine map and no activation: its mag
    |s| mag_conv + |t| is the value of the fused pass on absolute inputs."""
    x, w, b = rng.standard_normal((2, 7, 6, 4)), rng.standard_normal((3, 3, 4)), rng.standard_normal(4)
    s, t = rng.standard_normal(4), rng.standard_normal(4)
    _, mag = oracle.fwd_fused(x, w, b, post=(s, t, "none"), pad=1)
    ya, _ = oracle.fwd_fused(np.abs(x), np.abs(w), np.abs(b), post=(np.abs(s), np.abs(t), "none"), pad=1)
    assert np.array_equal(mag, ya)


# --------------------------------------- per-axis stride / dilation / padding

AXIS_CASES = [  # (N, H, W, C, FH, FW, (sh, sw), (dh, dw), (ph, pw))
    (2, 7, 9, 3, 3, 2, (1, 2), (2, 1), (2, 0)),
    (1, 6, 11, 2, 1, 5, (2, 1), (1, 2), (0, 4)),
    (2, 9, 5, 3, 4, 1, (3, 1), (1, 1), (1, 0)),
    (1, 8, 8, 2, 2, 3, (2, 3), (3, 1), (1, 2)),
    (1, 10, 7, 2, 3, 3, (2, 1), (1, 1), (1, 1)),
]


@pytest.mark.parametrize("case", AXIS_CASES)
def test_f64_axes_adjoint_and_transpose(case):
    """Per-axis parameters through the float64 loops: the adjoint identity
    holds exactly, and swapping H and W swaps the parameters of every pass."""
    N, H, W, C, FH, FW, S, D, P = case
    x, w, b = fint((N, H, W, C)), fint((FH, FW, C)), fint((C,))
    y, _ = oracle.fwd(x, w, None, S, D, P)
    dy = fint(y.shape)
    dx, _ = oracle.dgrad(dy, w, H, W, S, D, P)
    dw, _ = oracle.wgrad(x, dy, FH, FW, S, D, P)
    lhs = float(np.sum(y * dy))
    assert lhs == float(np.sum(x * dx)) == float(np.sum(w * dw))
    sw_ = lambda t: (t[1], t[0])  # noqa: E731
    xt, wt, dyt = x.transpose(0, 2, 1, 3), w.transpose(1, 0, 2), dy.transpose(0, 2, 1, 3)
    yb, _ = oracle.fwd(x, w, b, S, D, P)
    assert np.array_equal(yb, oracle.fwd(xt, wt, b, sw_(S), sw_(D), sw_(P))[0].transpose(0, 2, 1, 3))
    assert np.array_equal(dx, oracle.dgrad(dyt, wt, W, H, sw_(S), sw_(D), sw_(P))[0].transpose(0, 2, 1, 3))
    assert np.array_equal(dw, oracle.wgrad(xt, dyt, FW, FH, sw_(S), sw_(D), sw_(P))[0].transpose(1, 0, 2))


@pytest.mark.parametrize("case", AXIS_CASES)
def test_f64_axes_match_torch_autograd(case):
    N, H, W, C, FH, FW, S, D, P = case
    x, w, b = rng.standard_normal((N, H, W, C)), rng.standard_normal((FH, FW, C)), rng.standard_normal(C)
    xt, wt, yt = torch_dwconv(x, w, b, S, D, P)
    y, my = oracle.fwd(x, w, b, S, D, P)
    assert np.all(np.abs(y - yt.detach().permute(0, 2, 3, 1).numpy()) <= 1e-13 * (my + 1))
    dy = rng.standard_normal(y.shape)
    gx, gw = torch.autograd.grad(yt, (xt, wt), torch.from_numpy(dy).permute(0, 3, 1, 2))
    dx, mdx = oracle.dgrad(dy, w, H, W, S, D, P)
    dw, mdw = oracle.wgrad(x, dy, FH, FW, S, D, P)
    assert np.all(np.abs(dx - gx.permute(0, 2, 3, 1).numpy()) <= 1e-13 * (mdx + 1))
    assert np.all(np.abs(dw - gw.squeeze(1).permute(1, 2, 0).numpy()) <= 1e-13 * (mdw + 1))
