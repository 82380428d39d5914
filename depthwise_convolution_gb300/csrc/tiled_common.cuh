// Pieces shared by the register-tiled kernels (tiled_small.cu: forward and
// input gradient; tiled_wgrad.cu: weight gradient).
//
// A work unit is an output tile of NI images x (RT*TH) rows x (CT*TW)
// columns x 32 channels.  A CTA is 16 channel pairs x 8 thread tiles
// (NI*RT*CT = 8) = 128 threads; each thread owns one channel pair and a
// TH x TW block of outputs.  The unit's input halo -- (RT*TH-1)+FH rows by
// (CT*TW-1)+FW columns of the sub-grid, the "(T-1)S + (R-1)D + 1" extent of
// "Tiles, halos and partial sums" with S = D = 1 on the sub-grid -- is staged
// in shared memory with 16-byte cp.async copies; copies that fall outside the
// input use a zero source size, so padding is generated, never fetched.
#pragma once

#include <algorithm>

#include "common.cuh"

namespace dwc {
namespace tiled {

constexpr int kPairs = 16;                 // channel pairs per CTA (32 channels)
constexpr int kTiles = 8;                  // thread tiles per CTA
constexpr int kThreads = kPairs * kTiles;  // 128

struct Geo {
    int NI, RT, CT;        // thread tiles: images x rows x columns (product 8)
    int HH, HW;            // halo rows / columns per image
    int tiles_h, tiles_w;  // work units along output rows / columns
    int groups, ctiles;    // image groups (NI images each), channel tiles
    long long units;       // ctiles * groups * tiles_w * tiles_h
    long long per_ctile;   // groups * tiles_w * tiles_h
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_1() {
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");
}

// Unit index -> (channel tile, image group, column tile, row band); the row
// band varies fastest.
struct Unit {
    int ctile, group, twi, band;
};
__device__ __forceinline__ Unit decode(const Geo &g, long long u) {
    Unit r;
    r.ctile = (int)(u / g.per_ctile);
    long long v = u % g.per_ctile;
    r.band = (int)(v % g.tiles_h);
    v /= g.tiles_h;
    r.twi = (int)(v % g.tiles_w);
    r.group = (int)(v / g.tiles_w);
    return r;
}

// Stage the input halo of unit `un` into dst[NI][HH][HW][32] (zero outside).
template <typename T, int TH, int TW>
__device__ __forceinline__ void stage_halo(const TiledConv &p, const Geo &g, T *dst, const Unit &un) {
    constexpr int EPC = 16 / sizeof(T);  // elements per 16-byte copy
    constexpr int CPP = 32 / EPC;        // copies per pixel (32 channels)
    const T *in = static_cast<const T *>(p.in);
    const int ih0 = un.band * (g.RT * TH) - p.pad_h;
    const int iw0 = un.twi * (g.CT * TW) - p.pad_w;
    const int c0 = un.ctile * 32;
    const int total = g.NI * g.HH * g.HW * CPP;
    for (int k = threadIdx.x; k < total; k += kThreads) {
        const int q = k % CPP;
        const int pix = k / CPP;
        const int b = pix % g.HW;
        const int a = (pix / g.HW) % g.HH;
        const int il = pix / (g.HW * g.HH);
        const int nn = un.group * g.NI + il;
        const int ihs = ih0 + a, iws = iw0 + b, cc = c0 + q * EPC;
        const bool ok = nn < p.N && ihs >= 0 && ihs < p.Hs && iws >= 0 && iws < p.Ws && cc < p.C;
        const T *src = in;
        if (ok)
            src += (((long long)nn * p.Hf + (p.in_off + p.in_step * ihs)) * p.Wf +
                    (p.in_off + p.in_step * iws)) * (long long)p.C + cc;
        cp_async16(dst + (long long)pix * 32 + q * EPC, src, ok ? 16 : 0);
    }
}

// Stage the output-side tile of unit `un` (dy for the weight gradient) from
// `src` [N][OHs][OWs][C] into dst[NI][RT*TH][CT*TW][32] (zero outside).
template <typename T, int TH, int TW>
__device__ __forceinline__ void stage_out_tile(const TiledConv &p, const Geo &g, const T *src_base,
                                               T *dst, const Unit &un) {
    constexpr int EPC = 16 / sizeof(T);
    constexpr int CPP = 32 / EPC;
    const int rows = g.RT * TH, cols = g.CT * TW;
    const int i0 = un.band * rows, j0 = un.twi * cols;
    const int c0 = un.ctile * 32;
    const int total = g.NI * rows * cols * CPP;
    for (int k = threadIdx.x; k < total; k += kThreads) {
        const int q = k % CPP;
        const int pix = k / CPP;
        const int b = pix % cols;
        const int a = (pix / cols) % rows;
        const int il = pix / (cols * rows);
        const int nn = un.group * g.NI + il;
        const int i = i0 + a, j = j0 + b, cc = c0 + q * EPC;
        const bool ok = nn < p.N && i < p.OHs && j < p.OWs && cc < p.C;
        const T *src = src_base;
        if (ok) src += (((long long)nn * p.OHs + i) * p.OWs + j) * (long long)p.C + cc;
        cp_async16(dst + (long long)pix * 32 + q * EPC, src, ok ? 16 : 0);
    }
}

inline int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Thread-tile arrangement for an OHs x OWs output: columns first, then rows,
// then images, so that a CTA's 8 thread tiles stay busy on small maps.  The
// double-buffered stage (halo, plus the output-side tile when `out_tile`)
// is kept within `smem_cap` bytes.
inline Geo make_geo(const TiledConv &p, int TH, int TW, size_t elem, bool out_tile, size_t smem_cap) {
    Geo g{};
    auto arrange = [&](int CT) {
        g.CT = CT;
        g.RT = std::min(8 / g.CT, next_pow2((p.OHs + TH - 1) / TH));
        g.NI = 8 / (g.CT * g.RT);
        g.HH = g.RT * TH + p.FH - 1;
        g.HW = g.CT * TW + p.FW - 1;
    };
    auto stage_bytes = [&]() {
        size_t px = (size_t)g.HH * g.HW + (out_tile ? (size_t)g.RT * TH * g.CT * TW : 0);
        return 2 * (size_t)g.NI * px * 32 * elem;
    };
    arrange(std::min(8, next_pow2((p.OWs + TW - 1) / TW)));
    while (stage_bytes() > smem_cap && g.CT > 1) arrange(g.CT / 2);
    g.tiles_h = (p.OHs + g.RT * TH - 1) / (g.RT * TH);
    g.tiles_w = (p.OWs + g.CT * TW - 1) / (g.CT * TW);
    g.groups = (p.N + g.NI - 1) / g.NI;
    g.ctiles = (p.C + 31) / 32;
    g.per_ctile = (long long)g.groups * g.tiles_w * g.tiles_h;
    g.units = (long long)g.ctiles * g.per_ctile;
    return g;
}

inline size_t stage_bytes(const Geo &g, int TH, int TW, size_t elem, bool out_tile) {
    size_t px = (size_t)g.HH * g.HW + (out_tile ? (size_t)g.RT * TH * g.CT * TW : 0);
    return 2 * (size_t)g.NI * px * 32 * elem;
}

}  // namespace tiled
}  // namespace dwc
