// Register-tiled forward pass and input gradient for small filters (3x3, 5x5, 7x7).
//
// Design (the Flash-DWC §3.1-§3.4 dataflow restated for sm_103a):
//   * Work units, CTA shape and halo staging: see tiled_common.cuh.  Two
//     stage buffers: thread 0 issues the next unit's halo as one TMA tensor
//     copy while the CTA computes this one; mbarrier waits are bounded.
//   * The channel pair's FH x FW filter lives in registers (as stored) and
//     is reloaded only when the channel tile changes (filter reuse across all
//     spatial positions a thread computes, §3.2).
//   * Width-first register reuse (§3.3): the thread walks the TH+FH-1 input
//     rows of its window once; each row's TW+FW-1 values are read from shared
//     memory once, widened to fp32 once, and feed every (output row, filter
//     row) pair that uses that input row.  Multiply-adds accumulate in fp32
//     (Mac<T> in common.cuh: fma.rn.f32x2 for fp32 data, the mixed-precision
//     fma.rn.f32.{f16,bf16} on packed 16-bit pairs otherwise).
//   * Persistent grid: as many CTAs as fit on the SMs, each taking a
//     contiguous range of work units (ranges differ by at most one unit).
//   * Epilogue: bias added once (forward only), round to the storage type,
//     masked stores for spatial and channel tails; with zero_phases the other
//     output phases of each stride block are written as zeros.
#include "tiled_common.cuh"

namespace dwc {
namespace {

using namespace tiled;

// Tile choices per dtype class: thread tile TH x TW, CTAs per SM the register
// budget is sized for (MINB), and the cap on the double-buffered halo.
#ifndef DWCONV_S16_MINB
#define DWCONV_S16_MINB 4
#endif
#ifndef DWCONV_S16_SMEM_KB
#define DWCONV_S16_SMEM_KB 48
#endif
#ifndef DWCONV_S16_TH
#define DWCONV_S16_TH 2
#endif
#ifndef DWCONV_S16_TW
#define DWCONV_S16_TW 7
#endif

#ifndef DWCONV_S32_MINB
#define DWCONV_S32_MINB 3
#endif
#ifndef DWCONV_S32_SMEM_KB
#define DWCONV_S32_SMEM_KB 72
#endif
#ifndef DWCONV_S32_TH
#define DWCONV_S32_TH 2
#endif

// The register class decides the tile choice: packed 16-bit pairs, or pairs
// held as float2 (fp32 data, and FP8 data widened on load).
template <typename T> constexpr bool packed16() { return sizeof(typename Mac<T>::V) == 4; }

template <typename T>
size_t smem_cap() {
    return packed16<T>() ? DWCONV_S16_SMEM_KB * 1024 : DWCONV_S32_SMEM_KB * 1024;
}


// FUSE: the BN+Act prologue and the affine+activation epilogue of the fused
// forward pass (Flash-DWC §5.2) are compiled in -- 1: piecewise-linear
// activations only, 2: all; separate instances, so that the plain passes
// keep their own register allocation.
template <typename T, int FH, int FW, int TH, int TW, int MINB, int OS, int FUSE>
__global__ void __launch_bounds__(kThreads, MINB)
    tiled_small_kernel(const __grid_constant__ CUtensorMap halo_map, TiledConv p, Geo g, unsigned *err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2];
    constexpr int WW = TW + FW - 1;  // input columns one thread reads per row

    const int tid = threadIdx.x;
    const int cp = tid % kPairs;
    const int t = tid / kPairs;
    const int img_l = t / (g.RT * g.CT);
    const int rt = (t / g.CT) % g.RT;
    const int ct = t % g.CT;

    const unsigned box_bytes = halo_box_bytes(g, sizeof(T));
    const int halo_elems = g.HH * g.HW * 32;
    const unsigned buf_stride = align128(box_bytes);  // byte offset of stage buffer 1
    const T *wgt = static_cast<const T *>(p.w);
    using TO = typename OutOf<T>::type;
    TO *out = static_cast<TO *>(p.out);
    const int tile_rows = g.RT * TH, tile_cols = g.CT * TW;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    // One thread issues the whole halo of a unit as a single tensor copy.
    auto issue = [&](int u, int b) {
        const Unit un = decode(g, u);
        mbar_arrive_expect_tx(&bars[b], box_bytes);
        tma_load_4d(smem_raw + b * buf_stride, &halo_map, un.ctile * 32, un.twi * tile_cols - p.pad_w,
                    un.band * tile_rows - p.pad_h, un.group * g.NI, &bars[b]);
    };

    using M = Mac<T>;
    typename M::V wr[FH][FW];
    float2 bias2 = make_float2(0.f, 0.f);
    int loaded_ctile = -1;

    // Contiguous unit range per CTA (channel tile slowest: few filter reloads;
    // measured on GB300: 3 % faster for fp32 7x7 on 56x56 maps, 15 % on 14x14).
    const int u_end = (int)((long long)g.units * (blockIdx.x + 1) / gridDim.x);
    int u = (int)((long long)g.units * blockIdx.x / gridDim.x);
    if (tid == 0 && u < u_end) issue(u, 0);
    for (int k = 0; u < u_end; ++k, ++u) {
        const int un = u + 1 < u_end ? u + 1 : g.units;
        if (tid == 0 && un < g.units) issue(un, (k + 1) & 1);
        if (!mbar_wait(&bars[k & 1], (k >> 1) & 1)) {
            // Give up: record it, let the copy still in flight land, and leave.
            report_timeout(err);
            if (tid == 0 && un < g.units) mbar_wait(&bars[(k + 1) & 1], ((k + 1) >> 1) & 1);
            return;
        }

        const Unit cur = decode(g, u);
        const int c = cur.ctile * 32 + 2 * cp;
        const bool cvalid = c < p.C;
        if (FUSE && p.fz.pre()) {
            // BN+Act prologue, once per staged value, in place: thread (cp,
            // t) takes channel pair cp of every 8th halo row.  Positions
            // outside the input are padding of x' and stay zero; x' is
            // rounded to T as the unfused layer would store it.
            T *hb = reinterpret_cast<T *>(smem_raw + (k & 1) * buf_stride);
            const Affine a0 = cvalid ? affine_in(p.fz, c) : Affine{1.f, 0.f};
            const Affine a1 = cvalid ? affine_in(p.fz, c + 1) : Affine{1.f, 0.f};
            const float2 s2 = make_float2(a0.s, a1.s), t2 = make_float2(a0.t, a1.t);
            // Halo columns [c_lo, c_hi) lie inside the input.
            const int col_in = cur.twi * tile_cols - p.pad_w;
            const int c_lo = min(max(-col_in, 0), g.HW), c_hi = max(min(p.Ws - col_in, g.HW), c_lo);
            with_act<FUSE == 1>(p.fz.in_act, [&](auto act) {
                [[maybe_unused]] constexpr int A = decltype(act)::value;
#pragma unroll 1
                for (int rr = t; rr < g.NI * g.HH; rr += kTiles) {
                    const int im = rr / g.HH, r = rr - im * g.HH;
                    const int ih = cur.band * tile_rows - p.pad_h + r;
                    const bool rok = ih >= 0 && ih < p.Hs && cur.group * g.NI + im < p.N;
                    T *row = hb + rr * g.HW * 32 + 2 * cp;
                    const int lo = rok ? c_lo : g.HW, hi = rok ? c_hi : g.HW;
#pragma unroll 1
                    for (int col = 0; col < lo; ++col) Pair<T>::store(row + col * 32, make_float2(0.f, 0.f));
#pragma unroll 4
                    for (int col = lo; col < hi; ++col) {
                        if constexpr (sizeof(T) == 4) {
                            float2 *q = reinterpret_cast<float2 *>(row + col * 32);
                            *q = prologue_f32<A>(*q, s2, t2);
                        } else if constexpr (sizeof(T) == 2) {
                            unsigned *q = reinterpret_cast<unsigned *>(row + col * 32);
                            *q = prologue_packed<T, A>(*q, s2, t2);
                        }
                    }
#pragma unroll 1
                    for (int col = hi; col < g.HW; ++col) Pair<T>::store(row + col * 32, make_float2(0.f, 0.f));
                }
            });
            // The generic-proxy writes come before this buffer's next TMA
            // fill; every thread sees the whole transformed halo.
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            __syncthreads();
        }
        if (cur.ctile != loaded_ctile) {
            loaded_ctile = cur.ctile;
#pragma unroll
            for (int fh = 0; fh < FH; ++fh)
#pragma unroll
                for (int fw = 0; fw < FW; ++fw) {
                    const int sfh = p.flip ? FH - 1 - fh : fh;
                    const int sfw = p.flip ? FW - 1 - fw : fw;
                    wr[fh][fw] = cvalid ? M::load(wgt + (sfh * FW + sfw) * p.C + c) : M::zero();
                }
            bias2 = (p.bias && cvalid) ? make_float2(p.bias[c], p.bias[c + 1]) : make_float2(0.f, 0.f);
        }

        const T *s = reinterpret_cast<const T *>(smem_raw + (k & 1) * buf_stride) + img_l * halo_elems;
        const int r0 = rt * TH, j0 = ct * TW;
        float2 acc[TH][TW];
#pragma unroll
        for (int th = 0; th < TH; ++th)
#pragma unroll
            for (int tw = 0; tw < TW; ++tw) acc[th][tw] = bias2;

#pragma unroll
        for (int r = 0; r < TH + FH - 1; ++r) {
            typename M::V xv[WW];
            const T *srow = s + ((r0 + r) * g.HW + j0) * 32 + 2 * cp;
#pragma unroll
            for (int j = 0; j < WW; ++j) xv[j] = M::load(srow + j * 32);
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int fh = r - th;
                if (fh < 0 || fh >= FH) continue;
#pragma unroll
                for (int fw = 0; fw < FW; ++fw)
#pragma unroll
                    for (int tw = 0; tw < TW; ++tw)
                        M::fma(acc[th][tw], wr[fh][fw], xv[tw + fw]);
            }
        }

        const int n = cur.group * g.NI + img_l;
        if (FUSE && p.fz.post() && cvalid) {
            // Epilogue: per-channel affine map and activation on the fp32 sums.
            const Affine a0 = affine_out(p.fz, c), a1 = affine_out(p.fz, c + 1);
            with_act<FUSE == 1>(p.fz.out_act, [&](auto act) {
#pragma unroll
                for (int th = 0; th < TH; ++th)
#pragma unroll
                    for (int tw = 0; tw < TW; ++tw) {
                        acc[th][tw].x = activate(fmaf(a0.s, acc[th][tw].x, a0.t), decltype(act)::value);
                        acc[th][tw].y = activate(fmaf(a1.s, acc[th][tw].y, a1.t), decltype(act)::value);
                    }
            });
        }
        if (cvalid && n < p.N) {
            const int i0 = cur.band * tile_rows + r0;
            const int jj0 = cur.twi * tile_cols + j0;
            TO *img = out + (long long)n * p.OHf * p.OWf * p.C + c;
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int i = i0 + th;
                if (i >= p.OHs) break;
#pragma unroll
                for (int tw = 0; tw < TW; ++tw) {
                    const int j = jj0 + tw;
                    if (j >= p.OWs) break;
                    if (OS == 1) {
                        Pair<TO>::store(img + ((long long)i * p.OWf + j) * p.C, acc[th][tw]);
                    } else {
                        // Every position of the OS x OS block: the computed phase
                        // gets the sum, the others get zero.
#pragma unroll
                        for (int a = 0; a < OS; ++a)
#pragma unroll
                            for (int b = 0; b < OS; ++b) {
                                const int orow = OS * i + a, ocol = OS * j + b;
                                if (orow < p.OHf && ocol < p.OWf) {
                                    const bool hit = a == p.out_off_h && b == p.out_off_w;
                                    Pair<TO>::store(img + ((long long)orow * p.OWf + ocol) * p.C,
                                                   hit ? acc[th][tw] : make_float2(0.f, 0.f));
                                }
                            }
                    }
                }
            }
        }
        __syncthreads();  // this buffer is refilled by the copy issued next iteration
    }
}

template <typename T, int FH, int FW, int TH, int TW, int MINB, int OS, int FUSE = 0>
cudaError_t run(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    auto kern = tiled_small_kernel<T, FH, FW, TH, TW, MINB, OS, FUSE>;
    const Geo g = make_geo(p, TH, TW, sizeof(T), false, smem_cap<T>());
    if (g.units == 0) return cudaErrorNotSupported;
    const size_t smem = stage_bytes(g, TH, TW, sizeof(T), false);
    if (smem > 220 * 1024) return cudaErrorNotSupported;
    CUtensorMap map;
    if (!make_halo_map(&map, p, g, dt, sizeof(T))) return cudaErrorNotSupported;
    int per_sm = 0;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kThreads, smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const long long slots = (long long)sm_count() * per_sm;
    const int grid = (int)std::min<long long>(g.units, slots);
    kern<<<grid, kThreads, smem, st>>>(map, p, g, device_error_word());
    note_launches(1);
    note_kernel("tiled_small");
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_filter(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    constexpr bool k16 = packed16<T>();
    constexpr int TH7 = k16 ? DWCONV_S16_TH : DWCONV_S32_TH, TW7 = k16 ? DWCONV_S16_TW : 7;
    constexpr int MB7 = k16 ? DWCONV_S16_MINB : DWCONV_S32_MINB;
    if (p.zero_phases) {
        if (p.fz.pre() || p.fz.post()) return cudaErrorNotSupported;
        if (p.out_step_h != 2 || p.out_step_w != 2) return cudaErrorNotSupported;
        if (p.FH == 5 && p.FW == 5) return run<T, 5, 5, 4, 7, 2, 2>(p, dt, st);
        if (p.FH == 3 && p.FW == 3) return run<T, 3, 3, 4, 7, 3, 2>(p, dt, st);
        if (p.FH == 7 && p.FW == 7) return run<T, 7, 7, TH7, TW7, MB7, 2>(p, dt, st);
        return cudaErrorNotSupported;
    }
    if (p.out_step_h != 1 || p.out_step_w != 1) return cudaErrorNotSupported;
    if (p.fz.pre() || p.fz.post()) {
        if (p.flip) return cudaErrorNotSupported;
        // SiLU and GELU keep several values of their polynomial / exponential
        // live per output: those instances are sized for one CTA less per SM
        // (more registers per thread) so that nothing spills.
        if (!act_is_light(p.fz.in_act) || !act_is_light(p.fz.out_act)) {
            if (p.FH == 7 && p.FW == 7) return run<T, 7, 7, TH7, TW7, MB7 - 1, 1, 2>(p, dt, st);
            if (p.FH == 5 && p.FW == 5) return run<T, 5, 5, 4, 7, 1, 1, 2>(p, dt, st);
            if (p.FH == 3 && p.FW == 3) return run<T, 3, 3, 4, 7, 2, 1, 2>(p, dt, st);
            if (p.FH == 3 && p.FW == 5) return run<T, 3, 5, 4, 7, 2, 1, 2>(p, dt, st);
            return cudaErrorNotSupported;
        }
        if (p.FH == 7 && p.FW == 7) return run<T, 7, 7, TH7, TW7, MB7, 1, 1>(p, dt, st);
        if (p.FH == 5 && p.FW == 5) return run<T, 5, 5, 4, 7, 2, 1, 1>(p, dt, st);
        if (p.FH == 3 && p.FW == 3) return run<T, 3, 3, 4, 7, 3, 1, 1>(p, dt, st);
        if (p.FH == 3 && p.FW == 5) return run<T, 3, 5, 4, 7, 3, 1, 1>(p, dt, st);
        return cudaErrorNotSupported;
    }
    if (p.FH == 7 && p.FW == 7) return run<T, 7, 7, TH7, TW7, MB7, 1>(p, dt, st);
    if (p.FH == 5 && p.FW == 5) return run<T, 5, 5, 4, 7, 2, 1>(p, dt, st);
    if (p.FH == 3 && p.FW == 3) return run<T, 3, 3, 4, 7, 3, 1>(p, dt, st);
    if (p.FH == 3 && p.FW == 5) return run<T, 3, 5, 4, 7, 3, 1>(p, dt, st);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_tiled_small(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    switch (dt) {
        case DWCONV_FP32: return dispatch_filter<float>(p, dt, st);
        case DWCONV_FP16: return dispatch_filter<__half>(p, dt, st);
        case DWCONV_BF16: return dispatch_filter<__nv_bfloat16>(p, dt, st);
        case DWCONV_FP8_E4M3: return p.flip || p.fz.pre() ? cudaErrorNotSupported
                                                         : dispatch_filter<__nv_fp8_e4m3>(p, dt, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
