// Pieces shared by the register-tiled kernels (tiled_small.cu: forward and
// input gradient; tiled_wgrad.cu: weight gradient).
//
// A work unit is an output tile of NI images x (RT*TH) rows x (CT*TW)
// columns x 32 channels.  A CTA is 16 channel pairs x 8 thread tiles
// (NI*RT*CT = 8) = 128 threads; each thread owns one channel pair and a
// TH x TW block of outputs.  The unit's input halo -- (RT*TH-1)+FH rows by
// (CT*TW-1)+FW columns of the sub-grid, the "(T-1)S + (R-1)D + 1" extent of
// "Tiles, halos and partial sums" with S = D = 1 on the sub-grid -- is staged
// in shared memory by one TMA tensor copy issued by one thread; the copy
// engine fills everything outside the tensor with zeros, so padding is
// generated, never fetched.
#pragma once

#include <algorithm>

#include "common.cuh"
#include "tma.cuh"

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
    int units;             // ctiles * groups * tiles_w * tiles_h
    int per_ctile;         // groups * tiles_w * tiles_h
};

// Unit index -> (channel tile, image group, column tile, row band); the row
// band varies fastest.
struct Unit {
    int ctile, group, twi, band;
};
__device__ __forceinline__ Unit decode(const Geo &g, int u) {
    Unit r;
    r.ctile = u / g.per_ctile;
    int v = u - r.ctile * g.per_ctile;
    r.band = v % g.tiles_h;
    v /= g.tiles_h;
    r.twi = v % g.tiles_w;
    r.group = v / g.tiles_w;
    return r;
}

// Tensor map of the taps' sub-grid of p.in, [N][Hs][Ws][C] with the sub-grid
// steps folded into the strides; one box = one unit's halo [NI][HH][HW][32].
// Elements outside the sub-grid (padding, channel tail, missing images) are
// filled with zeros by the copy engine.
inline bool make_halo_map(CUtensorMap *m, const TiledConv &p, const Geo &g, dwconv_dtype dt, size_t es) {
    const char *base = static_cast<const char *>(p.in) + ((size_t)p.in_off_h * p.Wf + p.in_off_w) * p.C * es;
    const uint64_t dims[4] = {(uint64_t)p.C, (uint64_t)p.Ws, (uint64_t)p.Hs, (uint64_t)p.N};
    const uint64_t str[3] = {(uint64_t)p.in_step_w * p.C * es, (uint64_t)p.in_step_h * p.Wf * p.C * es,
                             (uint64_t)p.Hf * p.Wf * p.C * es};
    const uint32_t box[4] = {32, (uint32_t)g.HW, (uint32_t)g.HH, (uint32_t)g.NI};
    return encode_tmap_4d(m, dt, base, dims, str, box);
}

// Tensor map of an output-side tensor [N][OHs][OWs][C] (dy for the weight
// gradient); one box = one unit's output tile [NI][RT*TH][CT*TW][32].
inline bool make_tile_map(CUtensorMap *m, const void *base, const TiledConv &p, const Geo &g, int TH, int TW,
                          dwconv_dtype dt, size_t es) {
    const uint64_t dims[4] = {(uint64_t)p.C, (uint64_t)p.OWs, (uint64_t)p.OHs, (uint64_t)p.N};
    const uint64_t str[3] = {(uint64_t)p.C * es, (uint64_t)p.OWs * p.C * es, (uint64_t)p.OHs * p.OWs * p.C * es};
    const uint32_t box[4] = {32, (uint32_t)(g.CT * TW), (uint32_t)(g.RT * TH), (uint32_t)g.NI};
    return encode_tmap_4d(m, dt, base, dims, str, box);
}

// Bytes of one stage region, rounded up so the next region stays 128-byte aligned.
inline __host__ __device__ unsigned align128(unsigned b) { return (b + 127u) & ~127u; }

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
    const long long per = (long long)g.groups * g.tiles_w * g.tiles_h;
    const long long units = per * g.ctiles;
    g.per_ctile = (int)std::min<long long>(per, 1LL << 30);
    g.units = units < (1LL << 30) ? (int)units : 0;  // 0: too large for the tiled kernels
    return g;
}

// Bytes of one pipeline stage: the halo box, then (weight gradient) the tile box.
inline __host__ __device__ unsigned halo_box_bytes(const Geo &g, size_t elem) {
    return (unsigned)((size_t)g.NI * g.HH * g.HW * 32 * elem);
}
inline __host__ __device__ unsigned tile_box_bytes(const Geo &g, int TH, int TW, size_t elem) {
    return (unsigned)((size_t)g.NI * g.RT * TH * g.CT * TW * 32 * elem);
}
inline size_t stage_bytes(const Geo &g, int TH, int TW, size_t elem, bool out_tile) {
    return 2 * (size_t)(align128(halo_box_bytes(g, elem)) +
                        (out_tile ? align128(tile_box_bytes(g, TH, TW, elem)) : 0u));
}

}  // namespace tiled
}  // namespace dwc
