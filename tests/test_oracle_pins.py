"""Pins for the CPU oracle: what the pages print, closed forms, special cases,
brute force and an independent library, so that a mistake anywhere in the
oracle (a dropped term, a wrong sign or index, a transposed operand) fails.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import forms, pages

rng = np.random.default_rng(12345)


def rint(shape, lo=-9, hi=9):
    return rng.integers(lo, hi, size=shape, endpoint=True, dtype=np.int64)


def small_cases():
    """(N,H,W,C,FH,FW,S,D,P) over all stride/dilation/pad combos with OH, OW >= 1."""
    out = []
    for S, D in itertools.product((1, 2, 3), (1, 2)):
        for FH, FW in ((1, 1), (3, 3), (2, 3), (3, 1), (5, 4)):
            for P in range(0, D * (max(FH, FW) - 1) + 2):
                H, W = 7, 6
                if oracle.out_extent(H, FH, S, D, P) >= 1 and oracle.out_extent(W, FW, S, D, P) >= 1:
                    out.append((2, H, W, 3, FH, FW, S, D, P))
    return out


CASES = small_cases()


# ---------------------------------------------------------------- page values

def test_p2_storage_budget_worked_example(golden):
    g = golden("storage_budget.txt")
    b = pages.storage_budget(Th=2, Tw=2, Tc=2, Tm=2, R=3)
    assert pages.halo_extent(2, 1, 3, 1) == g["halo_rows"] == g["halo_cols"]
    assert b["input"] == g["input_bytes"]
    assert b["weights"] == g["weight_bytes"]
    assert b["partials"] == g["partial_bytes"]
    assert b["bias"] == g["bias_bytes"]
    assert b["total"] == g["total_bytes"]
    db = pages.storage_budget(Th=2, Tw=2, Tc=2, Tm=2, R=3, double_buffer=True)
    assert db["total"] == g["double_buffered_total"] > g["budget"]
    t1 = pages.storage_budget(Th=2, Tw=2, Tc=1, Tm=2, R=3, double_buffer=True)
    assert t1["input"] == g["tc1_input_bytes"]
    assert t1["weights"] == g["tc1_weight_bytes"]
    assert t1["total"] == g["tc1_double_buffered_total"] <= g["budget"]
    # The depthwise counterpart: one filter per channel, so Tc*R*R weight bytes.
    assert pages.storage_budget(2, 2, 2, 2, 3, depthwise=True)["weights"] == 18


def test_p1_p3_halo_extent_closed_form_and_brute_force(golden):
    g = golden("halo_span.txt")
    assert pages.halo_extent(g["s1_tile"], 1, g["s1_R"], 1) == g["s1_extent"]
    assert pages.halo_extent(g["s2_tile"], 2, g["s2_R"], 1) == g["s2_extent"]
    for T, S, D, R in itertools.product(range(1, 9), range(1, 4), range(1, 4), range(1, 8)):
        assert pages.halo_extent(T, S, R, D) == pages.touched_extent_brute(T, S, R, D)


@pytest.mark.parametrize("Th,S,D,R", [(2, 1, 1, 3), (2, 2, 1, 3), (3, 2, 2, 5), (4, 1, 3, 3), (1, 3, 2, 4)])
def test_p1_halo_matches_inputs_the_oracle_reads(Th, S, D, R):
    """The oracle's own index arithmetic: the inputs that an output tile depends
    on (found through the adjoint: dgrad of a tile indicator with an all-ones
    filter) span exactly halo_extent rows and columns."""
    H = W = 40
    P = 0
    OH = oracle.out_extent(H, R, S, D, P)
    dy = np.zeros((1, OH, OH, 1), dtype=np.int64)
    oh0 = 3
    dy[0, oh0:oh0 + Th, oh0:oh0 + Th, 0] = 1
    w = np.ones((R, R, 1), dtype=np.int64)
    dx, _ = oracle.dgrad(dy, w, H, W, S, D, P)
    rows, cols = np.nonzero(dx[0, :, :, 0])
    assert rows.max() - rows.min() + 1 == pages.halo_extent(Th, S, R, D)
    assert cols.max() - cols.min() + 1 == pages.halo_extent(Th, S, R, D)
    assert rows.min() == oh0 * S - P


def test_p4_tail_masking_page_numbers(golden):
    g = golden("masking.txt")
    tiles = pages.channel_tiles(g["M"], g["Tm"])
    assert len(tiles) == g["tiles"]
    assert tiles[-1] == g["last_tile_valid"]
    assert sum(tiles) == g["M"]


def test_p4_tail_masking_tiled_equals_untiled_c5():
    """C = 5 channels in tiles of 2: the masked tail tile changes nothing."""
    x, w, b = rint((1, 8, 8, 5), -128, 127), rint((3, 3, 5), -128, 127), rint((5,), -1000, 1000)
    y, _ = oracle.fwd(x, w, b, 1, 1, 1)
    yt = forms.tiled_fwd(x, w, b, 1, 1, 1, Th=3, Tw=3, Tc=2, row_groups=2)
    assert np.array_equal(y, yt)


def test_p5_traffic_model(golden):
    g = golden("traffic_model.txt")
    m, k, n, b = g["m"], g["k"], g["n"], g["b"]
    assert pages.q_min(m, k, n, b) == g["q_min"]
    assert pages.q_tile(m, k, n, b, 1) == g["q_tile_t1"]
    assert pages.q_tile(m, k, n, b, 2) == g["q_tile_t2"]
    for m, k, n, t in itertools.product((1, 2, 5, 8), (1, 3), (1, 4, 7), (1, 2, 3, 8)):
        assert pages.q_tile(m, k, n, 2, t) == pages.q_tile_simulated(m, k, n, 2, t)
        assert pages.q_tile(m, k, n, 2, t) >= pages.q_min(m, k, n, 2)
    # With one tile covering everything, the tiled traffic is the minimum.
    assert pages.q_tile(5, 3, 7, 4, 8) == pages.q_min(5, 3, 7, 4)


def test_p10_flashdwc_tile_model(golden):
    g = golden("flashdwc_tile_model.txt")
    assert round(pages.eta_filter_reuse(8), 2) == g["eta_filter_reuse_TM8"]
    assert round(pages.eta_block_filter(8, 32), 2) == g["eta_block_BN32_TM8"]
    assert round(pages.eta_gemv_limit(8, 32), 2) == g["eta_gemv_limit_BN32_TM8"]
    assert pages.eta_gemv(8, 10**9, 32) == pytest.approx(pages.eta_gemv_limit(8, 32), rel=1e-6)
    assert pages.toeplitz_k(8, 9) == 16
    assert pages.toeplitz_density(8, 9) == g["density_TM8_F9"]
    assert pages.toeplitz_density_brute(8, 9) == g["density_TM8_F9"]
    nz, tot = pages.toeplitz_nonzero_flops(16, 8, 9)
    assert (nz, tot) == (g["nonzero_flops"], g["total_flops"])
    assert pages.padded_filter_vector_len(9, 8) == g["padded_filter_len"]
    assert round(2 * pages.padded_filter_vector_len(9, 8) / 256, 2) == g["padded_filter_fraction"]
    assert nz / (256 + 128) == g["naive_gemm_intensity"]
    r = pages.width_first_loads(3, 3) / pages.rectangular_loads(3, 3)
    assert r == g["wf_over_rect_3x3"]
    for F in range(3, 52, 2):           # odd square filters, as the paper evaluates
        assert pages.width_first_loads(F, F) / pages.rectangular_loads(F, F) <= 1.25 + 1e-12
    assert pages.fragments_per_row(31) == g["fragments_FW31"]
    for TM, F in itertools.product(range(1, 12), range(1, 12)):
        assert pages.toeplitz_density(TM, F) == pytest.approx(pages.toeplitz_density_brute(TM, F))


# ------------------------------------------------- forms of the same operator

@pytest.mark.parametrize("case", CASES)
def test_p7_im2col_gemv_equals_direct_loop(case):
    N, H, W, C, FH, FW, S, D, P = case
    x, w, b = rint((N, H, W, C)), rint((FH, FW, C)), rint((C,))
    y, mag = oracle.fwd(x, w, b, S, D, P)
    assert np.array_equal(y, forms.im2col_gemv_fwd(x, w, b, S, D, P))
    assert np.all(mag >= np.abs(y))


@pytest.mark.parametrize("case", CASES[::3])
def test_p6_tiled_partial_sums_equal_untiled(case):
    N, H, W, C, FH, FW, S, D, P = case
    x, w, b = rint((N, H, W, C)), rint((FH, FW, C)), rint((C,))
    y, _ = oracle.fwd(x, w, b, S, D, P)
    for Th, Tw, Tc, groups in ((2, 2, 2, 2), (3, 1, 1, FH), (1, 4, 2, 1)):
        yt = forms.tiled_fwd(x, w, b, S, D, P, Th=Th, Tw=Tw, Tc=Tc, row_groups=min(groups, FH))
        assert np.array_equal(y, yt)
    # float64 on integer-valued data is exact as well
    yf, _ = oracle.fwd(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64), S, D, P)
    assert np.array_equal(yf, y.astype(np.float64))


def test_p6_bias_added_twice_is_caught():
    x, w, b = rint((1, 6, 6, 3)), rint((3, 3, 3)), rint((3,), 5, 9)
    y, _ = oracle.fwd(x, w, b, 1, 1, 1)
    bad = forms.tiled_fwd(x, w, b, 1, 1, 1, Th=2, Tw=2, Tc=2, row_groups=2, bias_mode="every_group")
    assert not np.array_equal(y, bad)
    assert np.array_equal(bad - y, np.broadcast_to(b, y.shape))


@pytest.mark.parametrize("case", CASES)
def test_p8_adjoint_identity_exact(case):
    """<fwd0(x,w), dy> = <x, dgrad(dy,w)> = <w, wgrad(x,dy)>, exactly in int64."""
    N, H, W, C, FH, FW, S, D, P = case
    x, w = rint((N, H, W, C)), rint((FH, FW, C))
    y, _ = oracle.fwd(x, w, None, S, D, P)
    dy = rint(y.shape)
    dx, _ = oracle.dgrad(dy, w, H, W, S, D, P)
    dw, _ = oracle.wgrad(x, dy, FH, FW, S, D, P)
    lhs = int(np.sum(y * dy))
    assert lhs == int(np.sum(x * dx))
    assert lhs == int(np.sum(w * dw))


@pytest.mark.parametrize("case", CASES[::3])
def test_dbias_is_the_adjoint_of_the_bias_term(case):
    """<fwd(x,w,b) - fwd(x,w,None), dy> = <b, dbias(dy)>, exactly in int64."""
    N, H, W, C, FH, FW, S, D, P = case
    x, w, b = rint((N, H, W, C)), rint((FH, FW, C)), rint((C,))
    y1, _ = oracle.fwd(x, w, b, S, D, P)
    y0, _ = oracle.fwd(x, w, None, S, D, P)
    dy = rint(y1.shape)
    db, mag = oracle.dbias(dy)
    assert int(np.sum((y1 - y0) * dy)) == int(np.sum(b * db))
    assert np.all(mag >= np.abs(db))


def test_dbias_closed_forms():
    dy = np.ones((3, 5, 4, 6), dtype=np.int64)
    db, mag = oracle.dbias(dy)
    assert np.array_equal(db, np.full(6, 60)) and np.array_equal(mag, db)
    alt = np.ones((2, 3, 3, 2), dtype=np.int64) * np.array([1, -1])   # channel 1 negative
    db, mag = oracle.dbias(alt)
    assert db.tolist() == [18, -18] and mag.tolist() == [18, 18]


@pytest.mark.parametrize("case", CASES[::2])
def test_dgrad_gather_form_equals_scatter_form(case):
    N, H, W, C, FH, FW, S, D, P = case
    w = rint((FH, FW, C))
    dy = rint((N, oracle.out_extent(H, FH, S, D, P), oracle.out_extent(W, FW, S, D, P), C))
    dx, mag = oracle.dgrad(dy, w, H, W, S, D, P)
    assert np.array_equal(dx, forms.dgrad_gather(dy, w, H, W, S, D, P))
    assert np.all(mag >= np.abs(dx))


# ------------------------------------------------------------- special cases

def test_p9_one_by_one_filter():
    x, w, b = rint((2, 5, 4, 3)), rint((1, 1, 3)), rint((3,))
    y, _ = oracle.fwd(x, w, b, 1, 1, 0)
    assert np.array_equal(y, x * w[0, 0] + b)
    y2, _ = oracle.fwd(x, w, b, 2, 1, 0)          # stride 2 subsamples
    assert np.array_equal(y2, x[:, ::2, ::2] * w[0, 0] + b)


@pytest.mark.parametrize("F,D", [(3, 1), (5, 1), (3, 2), (7, 3)])
def test_p9_centred_one_hot_is_identity(F, D):
    x, b = rint((2, 9, 8, 4)), rint((4,))
    w = np.zeros((F, F, 4), dtype=np.int64)
    w[F // 2, F // 2, :] = 1
    y, _ = oracle.fwd(x, w, b, 1, D, D * (F - 1) // 2)
    assert np.array_equal(y, x + b)


def test_p9_off_centre_one_hot_is_a_shift():
    x = rint((1, 9, 9, 2))
    w = np.zeros((3, 3, 2), dtype=np.int64)
    w[0, 2, :] = 1                                  # reads (oh-1, ow+1)
    y, _ = oracle.fwd(x, w, None, 1, 1, 1)
    expect = np.zeros_like(x)
    expect[:, 1:, :-1] = x[:, :-1, 1:]
    assert np.array_equal(y, expect)


def test_p9_constant_input_interior_and_corner():
    F, P = 5, 2
    x = np.full((1, 11, 11, 3), 3, dtype=np.int64)
    w, b = rint((F, F, 3)), rint((3,))
    y, _ = oracle.fwd(x, w, b, 1, 1, P)
    assert np.array_equal(y[0, 5, 5], b + 3 * w.sum(axis=(0, 1)))
    # The top-left corner sees only the taps with fh, fw >= P.
    assert np.array_equal(y[0, 0, 0], b + 3 * w[P:, P:].sum(axis=(0, 1)))


@pytest.mark.parametrize("F,D,P", [(3, 1, 1), (5, 1, 2), (3, 2, 2), (5, 2, 4), (7, 1, 3), (4, 1, 0)])
def test_p9_stride1_dgrad_is_forward_with_rotated_filter(F, D, P):
    H, W, C = 10, 9, 3
    w = rint((F, F, C))
    dy = rint((2, oracle.out_extent(H, F, 1, D, P), oracle.out_extent(W, F, 1, D, P), C))
    dx, _ = oracle.dgrad(dy, w, H, W, 1, D, P)
    assert np.array_equal(dx, forms.dgrad_rot180_stride1(dy, w, H, W, D, P))


def test_p9_stride2_dilation2_odd_positions_get_no_gradient():
    """5x5, stride 2, dilation 2, pad 4: every tap index is even, so dx is zero
    on odd rows and columns, and the forward pass never reads them."""
    H = W = 12
    w = rint((5, 5, 2))
    OH = oracle.out_extent(H, 5, 2, 2, 4)
    assert OH == 6
    dy = rint((1, OH, OH, 2))
    dx, _ = oracle.dgrad(dy, w, H, W, 2, 2, 4)
    assert not dx[:, 1::2, :].any() and not dx[:, :, 1::2].any()
    assert dx[:, ::2, ::2].any()
    x = rint((1, H, W, 2))
    x2 = x.copy()
    x2[:, 1::2] = 99
    x2[:, :, 1::2] = -99
    assert np.array_equal(oracle.fwd(x, w, None, 2, 2, 4)[0], oracle.fwd(x2, w, None, 2, 2, 4)[0])


def test_p9_one_dimensional_zero_padded_convolution():
    v = [3, 1, 4, 1, 5, 9, 2, 6]
    f = [2, -1, 7, 1, -3]
    expect = forms.conv1d_zero_pad(v, f)
    # np.convolve flips its kernel; DWC correlates, so feed it the reversed filter.
    assert expect == list(np.convolve(v, f[::-1], mode="same"))
    x = np.array(v, dtype=np.int64).reshape(1, 1, len(v), 1)
    w = np.array(f, dtype=np.int64).reshape(1, len(f), 1)
    y, _ = oracle.fwd(x, w, None, 1, 1, 2)
    # The symmetric pad of 2 also pads the single input row, giving OH = 5 output
    # rows; only the middle one (oh = 2) reads the real row, the rest read zeros.
    assert y.shape == (1, 5, len(v), 1)
    assert np.array_equal(y[0, 2, :, 0], expect)
    assert not np.delete(y[0, :, :, 0], 2, axis=0).any()


def test_output_extent_floor_convention():
    assert oracle.out_extent(112, 5, 2, 2, 4) == 56        # (112+8-8-1)//2 + 1
    assert oracle.out_extent(56, 7, 1, 1, 3) == 56
    assert oracle.out_extent(56, 31, 1, 1, 15) == 56
    assert oracle.out_extent(8, 3, 1, 1, 1) == 8
    assert oracle.out_extent(7, 3, 2, 1, 0) == 3           # (7-3)//2 + 1
    assert oracle.out_extent(2, 5, 1, 1, 0) <= 0


# ------------------------------------------------------ an independent library

@pytest.mark.parametrize("case", CASES[::4])
def test_p11_torch_conv2d_groups_float64(case):
    N, H, W, C, FH, FW, S, D, P = case
    x = rng.standard_normal((N, H, W, C))
    w = rng.standard_normal((FH, FW, C))
    b = rng.standard_normal(C)
    y, _ = oracle.fwd(x, w, b, S, D, P)
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w).permute(2, 0, 1).unsqueeze(1)
    yt = torch.nn.functional.conv2d(xt, wt, torch.from_numpy(b), stride=S, padding=P, dilation=D, groups=C)
    assert np.allclose(y, yt.permute(0, 2, 3, 1).numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- properties

def test_magnitude_equals_value_for_positive_data():
    x, w, b = rint((1, 6, 6, 2), 1, 5), rint((3, 3, 2), 1, 5), rint((2,), 1, 5)
    y, mag = oracle.fwd(x, w, b, 1, 1, 1)
    assert np.array_equal(y, mag)
    dy = rint(y.shape, 1, 5)
    dx, mdx = oracle.dgrad(dy, w, 6, 6, 1, 1, 1)
    dw, mdw = oracle.wgrad(x, dy, 3, 3, 1, 1, 1)
    assert np.array_equal(dx, mdx) and np.array_equal(dw, mdw)


def test_thread_count_does_not_change_results():
    x, w, b = rng.standard_normal((2, 9, 9, 7)), rng.standard_normal((3, 3, 7)), rng.standard_normal(7)
    y1, m1 = oracle.fwd(x, w, b, 1, 1, 1, nthreads=1)
    y4, m4 = oracle.fwd(x, w, b, 1, 1, 1, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(m1, m4)
    dy = rng.standard_normal(y1.shape)
    assert np.array_equal(oracle.wgrad(x, dy, 3, 3, 1, 1, 1, nthreads=1)[0],
                          oracle.wgrad(x, dy, 3, 3, 1, 1, 1, nthreads=5)[0])


def test_valid_tap_count_brute_force_matches_oracle():
    for (H, W, F, S, D, P) in ((9, 7, 3, 1, 1, 1), (12, 12, 5, 2, 2, 4), (7, 7, 7, 1, 1, 3), (10, 8, 3, 2, 1, 0)):
        x = np.ones((1, H, W, 1), dtype=np.int64)
        w = np.ones((F, F, 1), dtype=np.int64)
        y, _ = oracle.fwd(x, w, None, S, D, P)
        assert int(y.sum()) == forms.valid_tap_count(H, W, F, F, S, D, P)


def test_oracle_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.fwd(np.zeros((1, 2, 2, 1)), np.zeros((5, 5, 1)), None, 1, 1, 0)
    with pytest.raises(ValueError):
        oracle.fwd(np.zeros((1, 4, 4, 2)), np.zeros((3, 3, 3)), None, 1, 1, 1)


# ------------------------------------------------- per-axis stride/dilation/pad

AXIS_CASES = [  # (N, H, W, C, FH, FW, (sh, sw), (dh, dw), (ph, pw))
    (2, 7, 9, 3, 3, 2, (1, 2), (2, 1), (2, 0)),
    (1, 6, 11, 2, 1, 5, (2, 1), (1, 2), (0, 4)),
    (2, 9, 5, 3, 4, 1, (3, 1), (1, 1), (1, 0)),
    (1, 8, 8, 2, 2, 3, (2, 3), (3, 1), (1, 2)),
]


@pytest.mark.parametrize("case", AXIS_CASES)
def test_axes_swap_with_the_transpose(case):
    """Swapping H and W swaps the per-axis parameters: exact in int64 for all three passes."""
    N, H, W, C, FH, FW, S, D, P = case
    x, w, b = rint((N, H, W, C)), rint((FH, FW, C)), rint((C,))
    sw_ = lambda t: (t[1], t[0])  # noqa: E731
    xt, wt = x.transpose(0, 2, 1, 3), w.transpose(1, 0, 2)
    y, _ = oracle.fwd(x, w, b, S, D, P)
    yt, _ = oracle.fwd(xt, wt, b, sw_(S), sw_(D), sw_(P))
    assert np.array_equal(y, yt.transpose(0, 2, 1, 3))
    dy = rint(y.shape)
    dx, _ = oracle.dgrad(dy, w, H, W, S, D, P)
    dxt, _ = oracle.dgrad(dy.transpose(0, 2, 1, 3), wt, W, H, sw_(S), sw_(D), sw_(P))
    assert np.array_equal(dx, dxt.transpose(0, 2, 1, 3))
    dw, _ = oracle.wgrad(x, dy, FH, FW, S, D, P)
    dwt, _ = oracle.wgrad(xt, dy.transpose(0, 2, 1, 3), FW, FH, sw_(S), sw_(D), sw_(P))
    assert np.array_equal(dw, dwt.transpose(1, 0, 2))


@pytest.mark.parametrize("case", AXIS_CASES)
def test_axes_adjoint_identity_exact(case):
    N, H, W, C, FH, FW, S, D, P = case
    x, w = rint((N, H, W, C)), rint((FH, FW, C))
    y, _ = oracle.fwd(x, w, None, S, D, P)
    dy = rint(y.shape)
    dx, _ = oracle.dgrad(dy, w, H, W, S, D, P)
    dw, _ = oracle.wgrad(x, dy, FH, FW, S, D, P)
    lhs = int(np.sum(y * dy))
    assert lhs == int(np.sum(x * dx)) == int(np.sum(w * dw))


def test_strip_filter_is_a_1d_convolution_per_row():
    """A 1 x K filter with pad (0, K//2), row stride 2: every output row is the
    zero-padded 1-D convolution ("Outline of Programming Massively Parallel
    Processors", Convolution) of every other input row."""
    K = 5
    x, w = rint((2, 6, 10, 3)), rint((1, K, 3))
    y, _ = oracle.fwd(x, w, None, (2, 1), 1, (0, K // 2))
    assert y.shape == (2, 3, 10, 3)
    for n in range(2):
        for oh in range(3):
            for c in range(3):
                assert y[n, oh, :, c].tolist() == forms.conv1d_zero_pad(x[n, 2 * oh, :, c], w[0, :, c])


# ---------------------------------------------------------- fused epilogue

def test_activation_closed_forms():
    v = np.array([-7.0, -1.0, 0.0, 0.5, 3.0, 7.0])
    assert oracle.activation(v, "relu").tolist() == [0, 0, 0, 0.5, 3, 7]
    assert oracle.activation(v, "relu6").tolist() == [0, 0, 0, 0.5, 3, 6]
    assert oracle.activation(np.array([0.0]), "silu")[0] == 0 and oracle.activation(np.array([0.0]), "gelu")[0] == 0
    # x*f(x) - (-x)*f(-x) = x for f a symmetric CDF (sigmoid, Phi): act(x) - act(-x) = x
    x = np.linspace(-6, 6, 49)
    for act in ("relu", "silu", "gelu"):
        assert np.allclose(oracle.activation(x, act) - oracle.activation(-x, act), x, atol=1e-12)
    # GELU(1) = Phi(1) = 0.8413447460685429...; SiLU(1) = 1 / (1 + 1/e)
    assert abs(oracle.activation(np.array([1.0]), "gelu")[0] - 0.8413447460685429) < 1e-15
    assert abs(oracle.activation(np.array([1.0]), "silu")[0] - 1 / (1 + np.exp(-1.0))) < 1e-15


def test_fused_affine_without_activation_is_exact():
    x, w, b = rint((2, 7, 6, 4)), rint((3, 3, 4)), rint((4,))
    s, t = rint((4,), -3, 3), rint((4,))
    y, _ = oracle.fwd(x, w, b, 1, 1, 1)
    yf, mag = oracle.fwd_fused(x, w, b, post=(s, t, "none"), stride=1, dilation=1, pad=1)
    assert np.array_equal(yf, (s * y + t).astype(np.float64))
    assert np.all(mag >= np.abs(yf))
    yr, _ = oracle.fwd_fused(x, w, b, post=(s, t, "relu"), stride=1, dilation=1, pad=1)
    assert np.array_equal(yr, np.maximum(s * y + t, 0).astype(np.float64))


def test_round_to_matches_library_casts():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 5, 4000),
                        rng.standard_normal(200) * 1e-6])          # fp16 subnormals
    v = v[np.abs(v) < 65504]                                        # overflow is out of scope
    assert np.array_equal(oracle.round_to(v, "fp16"), v.astype(np.float16).astype(np.float64))
    assert np.array_equal(oracle.round_to(v, "fp32"), v.astype(np.float32).astype(np.float64))
    # bf16: from float32 values (one rounding either way), against torch's cast
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_to(v32.astype(np.float64), "bf16"), ref)
    # ties go to even: 1 + 2^-8 lies halfway between bf16 1 and 1 + 2^-7
    assert oracle.round_to(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]), "bf16").tolist() == [1.0, 1 + 2 * 2.0 ** -7]


def test_prologue_padding_stays_zero():
    # x' = act(0 * x + 5) = 5 inside the input; the padding of x' is zero, so a
    # 3x3 box filter gives 45 inside, 30 on an edge and 20 in a corner.
    x = np.zeros((1, 4, 5, 2))
    w = np.ones((3, 3, 2))
    y, _ = oracle.fwd_fused(x, w, pre=(np.zeros(2), np.full(2, 5.0), "none"), pad=1)
    assert y[0, 1, 1, 0] == 45 and y[0, 0, 2, 1] == 30 and y[0, 0, 0, 0] == 20 and y[0, 3, 4, 1] == 20
    # ReLU of a negative shift wipes the input: only the bias is left
    b = np.array([1.5, -2.0])
    y, _ = oracle.fwd_fused(rint((1, 4, 5, 2)), w, b, pre=(None, np.full(2, -100.0), "relu"), pad=1)
    assert np.all(y == b)


def test_prologue_affine_is_linear():
    # DWC(s x + t) = s DWC(x) + t DWC(1), with 1 the all-ones input (zero padded)
    x, w = rint((2, 6, 7, 3)), rint((3, 5, 3))
    s, t = rint((3,), -3, 3), rint((3,))
    for S, D, P in [(1, 1, (1, 2)), (2, 1, 2), (1, 2, 3)]:
        y, _ = oracle.fwd_fused(x, w, pre=(s, t, "none"), stride=S, dilation=D, pad=P)
        y1, _ = oracle.fwd(x, w, None, S, D, P)
        y0, _ = oracle.fwd(np.ones_like(x), w, None, S, D, P)
        assert np.array_equal(y, s * y1 + t * y0)


def test_prologue_rounds_to_storage_format():
    x = np.full((1, 3, 3, 1), 1.0)
    w = np.zeros((1, 1, 1)); w[0, 0, 0] = 1.0
    # 1 * 1 + 2^-9 rounds to 1 in bf16 (8 bits), stays in fp16 (11 bits)
    pre = (None, np.array([2.0 ** -9]), "none")
    assert np.all(oracle.fwd_fused(x, w, pre=pre, fmt="bf16")[0] == 1.0)
    assert np.all(oracle.fwd_fused(x, w, pre=pre, fmt="fp16")[0] == 1 + 2.0 ** -9)


# ---------------------------------------------------------------- FP8 E4M3

def test_e4m3_decode_known_codes():
    v = oracle.decode_e4m3(np.array([0x00, 0x38, 0xB8, 0x7E, 0x01, 0x08, 0x07, 0x40, 0x3C], dtype=np.uint8))
    assert v.tolist() == [0.0, 1.0, -1.0, 448.0, 2.0 ** -9, 2.0 ** -6, 7 * 2.0 ** -9, 2.0, 1.5]
    assert np.isnan(oracle.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # monotone over the positive codes 0x00..0x7E
    pos = got[:0x7F]
    assert np.all(np.diff(pos) > 0)
