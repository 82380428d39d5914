// Register-tiled forward pass and stride-1 input gradient for large filters
// (FW >= 8, e.g. 31x31), any FH x FW at run time.
//
// The filter of a 32-channel slab (FH*FW*32 values) no longer fits in
// registers, so the roles change relative to tiled_small.cu:
//   * The slab's whole filter is staged once in shared memory by one TMA
//     tensor copy and reloaded only when the CTA moves to another channel
//     tile (filter reuse across every output the CTA computes, Flash-DWC §3.2).
//   * Input rows stream through a ring of NS shared-memory slots, one TMA
//     copy per row with zero fill outside the input (padding generated).  A
//     CTA computes an output tile of RT*TH rows, so it walks RT*TH+FH-1 input
//     rows; each row feeds every (output row, filter row) pair that uses it.
//   * Warp-specialised pipeline: a ninth warp only issues copies; the eight
//     compute warps wait on per-slot "full" mbarriers and release slots on
//     "empty" mbarriers, so a warp whose output rows do not touch the current
//     input row moves on instead of idling at a CTA-wide barrier.  All waits
//     are bounded (tma.cuh).
//   * Width-first register reuse (§3.3, §3.4): for one input row a thread
//     slides a TW-wide register window along the filter width -- one new input
//     value per filter column -- and each filter value it reads from shared
//     memory feeds TW multiply-adds; TH output rows share each input value.
//   * CTA = 256 threads = 16 channel pairs x 16 thread tiles (NI images x RT
//     rows x CT columns of TH x TW tiles; the two tiles of a warp share a tile
//     row, so the filter reads of a warp are broadcasts).
//   * Persistent CTAs take contiguous ranges of work units (channel tile
//     slowest) so that filter reloads are rare.
#include "tiled_common.cuh"

namespace dwc {
namespace {

using namespace tiled;

constexpr int kLThreads = 256;
constexpr int kLTiles = kLThreads / kPairs;  // 16
// Thread tile TH x TW; DWCONV_L_FW31 also builds a fully unrolled 31-wide
// instance; DWCONV_L_SKIP_PAD_ROWS skips input rows that are all padding.
#ifndef DWCONV_L_TH
#define DWCONV_L_TH 2
#endif
#ifndef DWCONV_L_TW
#define DWCONV_L_TW 14
#endif
#ifndef DWCONV_L_FW31
#define DWCONV_L_FW31 0
#endif
#ifndef DWCONV_L_MAXR16
#define DWCONV_L_MAXR16 96
#endif
#ifndef DWCONV_L_NS
#define DWCONV_L_NS 8
#endif
#ifndef DWCONV_L_SKIP_PAD_ROWS
#define DWCONV_L_SKIP_PAD_ROWS 0
#endif

constexpr int kNS = DWCONV_L_NS;                       // input-row ring slots

struct GeoL {
    int NI, RT, CT;        // thread tiles: images x rows x columns (product 16)
    int HW;                // halo columns per image
    int R;                 // input rows walked per unit: RT*TH + FH - 1
    int tiles_h, tiles_w, groups, ctiles;
    int per_ctile, units;
    unsigned filt_bytes;   // FH*FW*32 elements
    unsigned row_bytes;    // NI*HW*32 elements
};

__device__ __forceinline__ Unit decode_l(const GeoL &g, int u) {
    Unit r;
    r.ctile = u / g.per_ctile;
    int v = u - r.ctile * g.per_ctile;
    r.band = v % g.tiles_h;
    v /= g.tiles_h;
    r.twi = v % g.tiles_w;
    r.group = v / g.tiles_w;
    return r;
}

// FWC: the filter width as a compile-time constant (0: read p.FW at run time).
// FLIP: the filter is read rotated by 180 degrees (stride-1 input gradient).
// MAXR: registers per thread, sized so the wanted number of 288-thread CTAs
// fits an SM: each of the 4 sub-partitions holds 16K registers, and two
// 9-warp CTAs put 5 warps on some sub-partition, so two CTAs need <= 102.
// FUSE: the affine+activation epilogue of the fused forward pass (Flash-DWC
// §5.2) is compiled in (this kernel provides no BN+Act prologue).
template <typename T, int TH, int TW, int MAXR, int FWC, bool FLIP, bool FUSE = false>
__global__ void __maxnreg__(MAXR)
    tiled_large_kernel(const __grid_constant__ CUtensorMap row_map, const __grid_constant__ CUtensorMap filt_map,
                       TiledConv p, GeoL g, unsigned *err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // full[s]: a row has landed in slot s; empty[s]: all consumer warps are done
    // with slot s; filt_full / filt_empty: the same for the filter slab.
    __shared__ __align__(8) uint64_t full[kNS], empty[kNS], filt_full, filt_empty;
    using M = Mac<T>;
    using V = typename M::V;
    constexpr int kConsumerWarps = kLThreads / 32;
    const int FW = FWC ? FWC : p.FW;

    const int tid = threadIdx.x;
    const unsigned slot_bytes = align128(g.row_bytes);
    unsigned char *ring = smem_raw + align128(g.filt_bytes);
    const int tile_rows = g.RT * TH, tile_cols = g.CT * TW;

    // Contiguous unit range of this CTA.
    const int u_begin = (int)((long long)g.units * blockIdx.x / gridDim.x);
    const int u_end = (int)((long long)g.units * (blockIdx.x + 1) / gridDim.x);

    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        mbar_init(&filt_full, 1);
        mbar_init(&filt_empty, kConsumerWarps);
        mbar_fence_init();
    }
    __syncthreads();

    if (tid >= kLThreads) {  // ---------------- producer warp: one lane issues all copies
        if (tid != kLThreads) return;
        int q = 0, loaded = -1, reloads = 0;
        for (int u = u_begin; u < u_end; ++u) {
            const Unit un = decode_l(g, u);
            if (un.ctile != loaded) {
                if (reloads > 0 && !mbar_wait(&filt_empty, (reloads - 1) & 1)) {
                    report_timeout(err);
                    return;
                }
                mbar_arrive_expect_tx(&filt_full, g.filt_bytes);
                tma_load_4d(smem_raw, &filt_map, un.ctile * 32, 0, 0, 0, &filt_full);
                loaded = un.ctile;
                ++reloads;
            }
            for (int r = 0; r < g.R; ++r, ++q) {
                const int s = q % kNS, k = q / kNS;
                if (k > 0 && !mbar_wait(&empty[s], (k - 1) & 1)) {
                    report_timeout(err);
                    return;
                }
                mbar_arrive_expect_tx(&full[s], g.row_bytes);
                tma_load_4d(ring + s * slot_bytes, &row_map, un.ctile * 32, un.twi * tile_cols - p.pad_w,
                            un.band * tile_rows - p.pad_h + r, un.group * g.NI, &full[s]);
            }
        }
        return;
    }

    // ---------------------------------------- consumer warps
    const int lane = tid % 32;
    const int cp = tid % kPairs;
    const int t = tid / kPairs;
    const int ct = t % g.CT;
    const int rt = (t / g.CT) % g.RT;
    const int img_l = t / (g.CT * g.RT);
    const T *filt = reinterpret_cast<const T *>(smem_raw);
    T *out = static_cast<T *>(p.out);

    int q = 0, loaded = -1, filt_seen = 0;
    for (int u = u_begin; u < u_end; ++u) {
        const Unit cur = decode_l(g, u);
        if (cur.ctile != loaded) {
            if (!mbar_wait(&filt_full, filt_seen & 1)) {
                report_timeout(err);
                return;
            }
            ++filt_seen;
            loaded = cur.ctile;
        }
        const int c = cur.ctile * 32 + 2 * cp;
        const float2 bias2 =
            (p.bias && c < p.C) ? make_float2(p.bias[c], p.bias[c + 1]) : make_float2(0.f, 0.f);
        float2 acc[TH][TW];
#pragma unroll
        for (int th = 0; th < TH; ++th)
#pragma unroll
            for (int tw = 0; tw < TW; ++tw) acc[th][tw] = bias2;

        for (int r = 0; r < g.R; ++r, ++q) {
            const int s = q % kNS;
            // Filter rows this thread's output rows need from input row r; rows
            // outside the input are all padding and contribute nothing.
            const int fh0 = r - rt * TH;  // filter row of output row th = 0
            bool any = false;
#pragma unroll
            for (int th = 0; th < TH; ++th) any |= (fh0 - th >= 0 && fh0 - th < p.FH);
#if DWCONV_L_SKIP_PAD_ROWS
            const int in_row = cur.band * tile_rows - p.pad_h + r;
            any = any && in_row >= 0 && in_row < p.Hs;
#endif
            if (any) {
                if (!mbar_wait(&full[s], (q / kNS) & 1)) {
                    report_timeout(err);
                    return;
                }
                const T *xrow = reinterpret_cast<const T *>(ring + s * slot_bytes) +
                                (img_l * g.HW + ct * TW) * 32 + 2 * cp;
                const T *wrow[TH];
                bool valid[TH];
#pragma unroll
                for (int th = 0; th < TH; ++th) {
                    const int fh = fh0 - th;
                    valid[th] = fh >= 0 && fh < p.FH;
                    const int sfh = FLIP ? p.FH - 1 - fh : fh;
                    // Row start; with FLIP the row is walked backwards from its end.
                    wrow[th] = filt + ((valid[th] ? sfh : 0) * FW + (FLIP ? FW - 1 : 0)) * 32 + 2 * cp;
                }
                V xw[TW];
#pragma unroll
                for (int k = 0; k < TW; ++k) xw[k] = M::load(xrow + k * 32);
                // Filter columns in blocks of TW so the window slot of each input
                // value is a compile-time index.
                for (int fb = 0; fb < FW; fb += TW) {
#pragma unroll
                    for (int k = 0; k < TW; ++k) {
                        const int fw = fb + k;
                        if (fw < FW) {
                            const int off = (FLIP ? -fw : fw) * 32;
                            V wv[TH];
#pragma unroll
                            for (int th = 0; th < TH; ++th) wv[th] = valid[th] ? M::load(wrow[th] + off) : M::zero();
#pragma unroll
                            for (int th = 0; th < TH; ++th)
#pragma unroll
                                for (int tw = 0; tw < TW; ++tw) M::fma(acc[th][tw], wv[th], xw[(tw + k) % TW]);
                            // x[fw] is no longer needed; its slot takes x[fw + TW].
                            if (fw + TW < TW + FW - 1) xw[k] = M::load(xrow + (fw + TW) * 32);
                        }
                    }
                }
            } else if (!mbar_wait(&full[s], (q / kNS) & 1)) {
                // Not needed by this warp, but wait for it so that no warp runs
                // more than a ring ahead of the slowest one.
                report_timeout(err);
                return;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // Unit done: store, and release the filter if the next unit needs another.
        const int n = cur.group * g.NI + img_l;
        if (FUSE && p.fz.post() && c < p.C) {
            const Affine a0 = affine_out(p.fz, c), a1 = affine_out(p.fz, c + 1);
            with_act(p.fz.out_act, [&](auto act) {
#pragma unroll
                for (int th = 0; th < TH; ++th)
#pragma unroll
                    for (int tw = 0; tw < TW; ++tw) {
                        acc[th][tw].x = activate(fmaf(a0.s, acc[th][tw].x, a0.t), decltype(act)::value);
                        acc[th][tw].y = activate(fmaf(a1.s, acc[th][tw].y, a1.t), decltype(act)::value);
                    }
            });
        }
        if (c < p.C && n < p.N) {
            const int i0 = cur.band * tile_rows + rt * TH;
            const int j0 = cur.twi * tile_cols + ct * TW;
            T *img = out + (long long)n * p.OHf * p.OWf * p.C + c;
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int i = i0 + th;
                if (i >= p.OHs) break;
#pragma unroll
                for (int tw = 0; tw < TW; ++tw) {
                    const int j = j0 + tw;
                    if (j >= p.OWs) break;
                    const long long px = p.transpose ? (long long)j * p.OWf + i : (long long)i * p.OWf + j;
                    Pair<T>::store(img + px * p.C, acc[th][tw]);
                }
            }
        }
        if (u + 1 < u_end && decode_l(g, u + 1).ctile != cur.ctile) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&filt_empty);
        }
    }
}

template <typename T, int TH, int TW>
bool plan(const TiledConv &p, GeoL &g, size_t &smem) {
    g = GeoL{};
    auto arrange = [&](int CT) {
        g.CT = CT;
        g.RT = std::min(kLTiles / g.CT, next_pow2((p.OHs + TH - 1) / TH));
        g.NI = kLTiles / (g.CT * g.RT);
    };
    arrange(std::min(kLTiles, next_pow2((p.OWs + TW - 1) / TW)));
    g.HW = g.CT * TW + p.FW - 1;
    g.R = g.RT * TH + p.FH - 1;
    g.tiles_h = (p.OHs + g.RT * TH - 1) / (g.RT * TH);
    g.tiles_w = (p.OWs + g.CT * TW - 1) / (g.CT * TW);
    g.groups = (p.N + g.NI - 1) / g.NI;
    g.ctiles = (p.C + 31) / 32;
    const long long per = (long long)g.groups * g.tiles_w * g.tiles_h;
    if (per * g.ctiles >= (1LL << 30) || per * g.ctiles * g.R >= (1LL << 31)) return false;
    g.per_ctile = (int)per;
    g.units = (int)(per * g.ctiles);
    g.filt_bytes = (unsigned)((size_t)p.FH * p.FW * 32 * sizeof(T));
    g.row_bytes = (unsigned)((size_t)g.NI * g.HW * 32 * sizeof(T));
    if (p.FH > 256 || p.FW > 256 || g.HW > 256) return false;  // TMA box limits
    smem = align128(g.filt_bytes) + (size_t)kNS * align128(g.row_bytes);
    return smem <= 220 * 1024;
}

template <typename T, int TH, int TW, int MAXR, int FWC, bool FLIP, bool FUSE = false>
cudaError_t run(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    GeoL g;
    size_t smem;
    if (!plan<T, TH, TW>(p, g, smem)) return cudaErrorNotSupported;
    // Input rows: the taps' sub-grid of p.in, one row of the unit's halo per box.
    const size_t es = sizeof(T);
    const char *base = static_cast<const char *>(p.in) + ((size_t)p.in_off_h * p.Wf + p.in_off_w) * p.C * es;
    const uint64_t dims[4] = {(uint64_t)p.C, (uint64_t)p.Ws, (uint64_t)p.Hs, (uint64_t)p.N};
    uint64_t str[3];
    in_strides(p, es, str);
    const uint32_t box[4] = {32, (uint32_t)g.HW, 1, (uint32_t)g.NI};
    // Filter [FH][FW][C] as a 4-D tensor with a unit outer dimension; one box =
    // the whole filter of a 32-channel slab.
    const uint64_t fdims[4] = {(uint64_t)p.C, (uint64_t)p.FW, (uint64_t)p.FH, 1};
    // Transposed view: the kernel's filter column fw is memory row fw, whose
    // stride is FH (the memory width) * C elements.
    const uint64_t fstr[3] = {(uint64_t)(p.transpose ? p.FH : 1) * p.C * es,
                              (uint64_t)(p.transpose ? 1 : p.FW) * p.C * es, (uint64_t)p.FH * p.FW * p.C * es};
    const uint32_t fbox[4] = {32, (uint32_t)p.FW, (uint32_t)p.FH, 1};
    CUtensorMap row_map, filt_map;
    if (!encode_tmap_4d(&row_map, dt, base, dims, str, box) ||
        !encode_tmap_4d(&filt_map, dt, p.w, fdims, fstr, fbox))
        return cudaErrorNotSupported;
    auto kern = tiled_large_kernel<T, TH, TW, MAXR, FWC, FLIP, FUSE>;
    int per_sm = 0;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kLThreads + 32, smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const long long slots = (long long)sm_count() * per_sm;
    const int grid = (int)std::min<long long>(g.units, slots);
    kern<<<grid, kLThreads + 32, smem, st>>>(row_map, filt_map, p, g, device_error_word());
    note_launches(1);
    note_kernel("tiled_large");
    return cudaGetLastError();
}

}  // namespace

template <typename T, int MAXR>
cudaError_t by_width(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    constexpr int TH = DWCONV_L_TH, TW = DWCONV_L_TW;
#if DWCONV_L_FW31
    if (p.FW == 31 && !p.fz.pre() && !p.fz.post()) return p.flip ? run<T, TH, TW, MAXR, 31, true>(p, dt, st) : run<T, TH, TW, MAXR, 31, false>(p, dt, st);
#endif
    if (p.fz.pre()) return cudaErrorNotSupported;
    // Nine warps per CTA put three on one SM sub-partition, whose register
    // file holds 16384: at most 170 registers per thread.
    constexpr int kMaxR = MAXR < 168 ? MAXR : 168;
    if (p.fz.post()) return p.flip ? cudaErrorNotSupported : run<T, TH, TW, kMaxR, 0, false, true>(p, dt, st);
    return p.flip ? run<T, TH, TW, MAXR, 0, true>(p, dt, st) : run<T, TH, TW, MAXR, 0, false>(p, dt, st);
}

cudaError_t launch_tiled_large(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (p.FW < 8 || p.zero_phases || p.out_step_h != 1 || p.out_step_w != 1) return cudaErrorNotSupported;
    switch (dt) {
        case DWCONV_FP32: return by_width<float, 224>(p, dt, st);
        case DWCONV_FP16: return by_width<__half, DWCONV_L_MAXR16>(p, dt, st);
        case DWCONV_BF16: return by_width<__nv_bfloat16, DWCONV_L_MAXR16>(p, dt, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
