"""Arithmetic the pages print, written out as plain functions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Each helper cites the
passage it restates; ``tests/test_oracle_pins.py`` checks every one against
the numbers the pages print and against brute force.
"""
from __future__ import annotations

import math


# --- "Tiles, halos and partial sums", section "Partition tensors to fit storage"

def halo_extent(T: int, S: int, R: int, D: int) -> int:
    """Input rows (or columns) an output tile of T rows needs.

    Stride S, dilation D, kernel extent R: (T-1)*S + (R-1)*D + 1.
    """
    return (T - 1) * S + (R - 1) * D + 1


def touched_extent_brute(T: int, S: int, R: int, D: int) -> int:
    """Same quantity by enumeration: span of {t*S + r*D} over t<T, r<R."""
    idx = {t * S + r * D for t in range(T) for r in range(R)}
    return max(idx) - min(idx) + 1


# --- "Tiles, halos and partial sums", section "Worked storage budget"

def storage_budget(Th, Tw, Tc, Tm, R, S=1, D=1, in_bytes=1, w_bytes=1, psum_bytes=4,
                   bias_bytes=4, double_buffer=False, depthwise=False):
    """On-chip bytes of one tile of a convolution, as the worked budget counts them.

    input    = halo_h * halo_w * Tc * in_bytes
    weights  = Tc * Tm * R * R * w_bytes   (general convolution)
             = Tc * R * R * w_bytes        (depthwise: each channel one filter)
    partials = Th * Tw * Tm * psum_bytes
    bias     = Tm * bias_bytes
    Double-buffering duplicates input and weights only; partial sums and bias
    stay single.  Scales, addresses and control storage are excluded, as the
    page says.
    """
    hh, hw = halo_extent(Th, S, R, D), halo_extent(Tw, S, R, D)
    inp = hh * hw * Tc * in_bytes
    wts = (Tc * R * R if depthwise else Tc * Tm * R * R) * w_bytes
    ps = Th * Tw * Tm * psum_bytes
    bias = Tm * bias_bytes
    total = (2 if double_buffer else 1) * (inp + wts) + ps + bias
    return {"input": inp, "weights": wts, "partials": ps, "bias": bias, "total": total}


def channel_tiles(M: int, Tm: int):
    """Valid channels in each of the ceil(M/Tm) output-channel tiles (tail masked)."""
    return [min(Tm, M - t * Tm) for t in range((M + Tm - 1) // Tm)]


# --- "10.5 Why data reuse matters" (GEMM traffic model, beta = 0)

def q_min(m: int, k: int, n: int, b: int) -> int:
    """Ideal traffic of C = AB: read A and B once, write C once: (mk+kn+mn)*b."""
    return (m * k + k * n + m * n) * b


def q_tile(m: int, k: int, n: int, b: int, t: int) -> int:
    """Traffic with t x t output tiles and no reuse between output tiles.

    b * (mk*ceil(n/t) + kn*ceil(m/t) + mn).
    """
    return b * (m * k * math.ceil(n / t) + k * n * math.ceil(m / t) + m * n)


def q_tile_simulated(m: int, k: int, n: int, b: int, t: int) -> int:
    """Brute-force count of the same traffic: walk the output tiles, load the
    A rows and B columns each tile needs, store the tile."""
    total = 0
    for i0 in range(0, m, t):
        rows = min(t, m - i0)
        for j0 in range(0, n, t):
            cols = min(t, n - j0)
            total += rows * k * b      # the A rows of this tile
            total += k * cols * b      # the B columns of this tile
            total += rows * cols * b   # the C tile, written once
    return total


# --- Flash-DWC §3.2-§3.4 and §4.2-§4.3 tile-model closed forms (elements, not bytes)

def eta_filter_reuse(TM: int) -> float:
    """§3.2: one filter element loaded per TM FMAs over TM inputs: 2TM/(TM+1)."""
    return 2 * TM / (TM + 1)


def eta_block_filter(TM: int, BN: int) -> float:
    """§3.2: the filter fragment shared by 512/BN threads in shared memory."""
    return 2 * TM / (TM + BN / 512)


def eta_gemv(TM: int, FW: int, BN: int) -> float:
    """§3.4: with width-first reuse, 2TM / (1 + (TM-1)/FW + BN/512)."""
    return 2 * TM / (1 + (TM - 1) / FW + BN / 512)


def eta_gemv_limit(TM: int, BN: int) -> float:
    """§3.4: the FW -> infinity limit of eta_gemv."""
    return 2 * TM / (1 + BN / 512)


def width_first_loads(FH: int, FW: int, TM: int = 8) -> int:
    """§3.3: inputs loaded by width-first reuse for TM outputs (square filters)."""
    return FW * (FH + TM - 1)


def rectangular_loads(FH: int, FW: int) -> int:
    """§3.3: inputs loaded by the 2x4 rectangular reuse."""
    return (FW + 2 - 1) * (FH + 4 - 1)


def toeplitz_k(TM: int, F_frag: int) -> int:
    """§4.2: rows of the filter matrix, K = TM + F_frag - 1."""
    return TM + F_frag - 1


def toeplitz_density(TM: int, F_frag: int) -> float:
    """§4.2: fraction of non-zero entries of the K x TM filter matrix, F_frag/K."""
    return F_frag / toeplitz_k(TM, F_frag)


def toeplitz_nonzero_flops(M: int, TM: int, F_frag: int):
    """§4.2: (non-zero, total) multiply-add flops of one packed M x K x TM GEMM."""
    K = toeplitz_k(TM, F_frag)
    return 2 * M * TM * F_frag, 2 * M * TM * K


def toeplitz_density_brute(TM: int, F_frag: int) -> float:
    """Density by building the filter matrix: column i holds the fragment from row i."""
    K = toeplitz_k(TM, F_frag)
    nz = 0
    for col in range(TM):
        for row in range(K):
            if col <= row < col + F_frag:
                nz += 1
    return nz / (K * TM)


def padded_filter_vector_len(F_frag: int, TM: int) -> int:
    """§4.3: the fragment with TM-1 zeros on each side."""
    return F_frag + 2 * (TM - 1)


def fragments_per_row(FW: int, F_frag: int = 9) -> int:
    """§4.2: a filter row splits into ceil(FW/9) width-9 fragments."""
    return math.ceil(FW / F_frag)
