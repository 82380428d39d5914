// Register-tiled weight gradient for small filters (Flash-DWC §5.1, "BFC").
//
//   dw[fh,fw,c] = sum over (n, i, j) of dy[n,i,j,c] * x_sub[n, i - pad + fh, j - pad + fw, c]
//
// on the same sub-grid description as the forward pass (tiled_common.cuh).
// The output dw is tiny (FH*FW*C) while the accumulation axis N*OH*OW is
// long, so the work is split along the accumulation axis (§5.1
// "accumulation-axis parallelisation"):
//   * grid = channel tiles x Zc; CTA (ctile, z) takes the work units
//     z, z + Zc, z + 2 Zc, ... of its channel tile; one thread stages each
//     unit's x halo and dy tile in shared memory with two TMA tensor copies on
//     one mbarrier (double-buffered, bounded waits);
//   * every thread keeps the FH x FW fp32 accumulators of its channel pair in
//     registers for the whole CTA, and walks its window row-stationary: each
//     x row is read once and feeds every (dy row, filter row) pair using it;
//     multiply-adds accumulate in fp32 (Mac<T> in common.cuh);
//   * at the end the 8 thread tiles sharing a channel pair are summed with a
//     warp shuffle and a fixed-order pass through shared memory, and the CTA
//     writes part[z][fh*FW+fw][c];
//   * wgrad_reduce (direct.cu) then sums the Zc slices in a fixed order, so
//     the result is bit-identical from call to call (no atomics).
#include "tiled_common.cuh"

namespace dwc {
namespace {

using namespace tiled;

// Tile choices for 16-bit data: thread tile TH x TW, CTAs per SM the
// register budget is sized for (MINB), cap on the double-buffered stage.
#ifndef DWCONV_W16_MINB
#define DWCONV_W16_MINB 3
#endif
#ifndef DWCONV_W16_SMEM_KB
#define DWCONV_W16_SMEM_KB 72
#endif
#ifndef DWCONV_W16_TH
#define DWCONV_W16_TH 2
#endif
#ifndef DWCONV_W16_TW
#define DWCONV_W16_TW 7
#endif

// 16-bit data, filter height DWCONV_W_FFMA2_FH: widen on load and use packed
// fp32 FMAs (MacW).  Measured on GB300: faster for the 5x5 layer (4x7 thread
// tiles, 0.033 against 0.035 ms), slower for 7x7 (0.099 against 0.083 ms).
#ifndef DWCONV_W_FFMA2_FH
#define DWCONV_W_FFMA2_FH 5
#endif

// CTAs per SM the 7x7 hybrid-accumulation instance is sized for (its fp16
// partial sums add FH*FW registers to the fp32 accumulators).
#ifndef DWCONV_WHA_MINB
#define DWCONV_WHA_MINB 3
#endif


// HA (fp16 data only): hybrid accumulation, the opt-in of Flash-DWC §5.1
// "mixed accumulation" -- each thread's TH x TW products of a unit are summed
// per tap in fp16 (packed HFMA2, two channels per instruction), and that
// partial sum is added to the fp32 accumulator once per unit.
template <typename T, int FH, int FW, int TH, int TW, int MINB, bool HA = false>
__global__ void __launch_bounds__(kThreads, MINB)
    tiled_wgrad_kernel(const __grid_constant__ CUtensorMap halo_map, const __grid_constant__ CUtensorMap dy_map,
                       TiledConv p, Geo g, float *__restrict__ part, int Zc, unsigned *err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2];
    constexpr int WW = TW + FW - 1;

    const int tid = threadIdx.x;
    const int cp = tid % kPairs;
    const int t = tid / kPairs;
    const int img_l = t / (g.RT * g.CT);
    const int rt = (t / g.CT) % g.RT;
    const int ct = t % g.CT;

    const int tile_rows = g.RT * TH, tile_cols = g.CT * TW;
    const int halo_elems = g.HH * g.HW * 32;
    const int otile_elems = tile_rows * tile_cols * 32;
    const unsigned hb = halo_box_bytes(g, sizeof(T)), tb = tile_box_bytes(g, TH, TW, sizeof(T));
    const unsigned stage = align128(hb) + align128(tb);

    const int ctile = blockIdx.x / Zc;
    const int z = blockIdx.x % Zc;
    const int base = ctile * g.per_ctile;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    // One thread issues both boxes of a unit (x halo, dy tile) on one barrier.
    auto issue = [&](int v, int b) {
        const Unit un = decode(g, base + v);
        mbar_arrive_expect_tx(&bars[b], hb + tb);
        unsigned char *dst = smem_raw + b * stage;
        tma_load_4d(dst, &halo_map, un.ctile * 32, un.twi * tile_cols - p.pad_w,
                    un.band * tile_rows - p.pad_h, un.group * g.NI, &bars[b]);
        tma_load_4d(dst + align128(hb), &dy_map, un.ctile * 32, un.twi * tile_cols, un.band * tile_rows,
                    un.group * g.NI, &bars[b]);
    };

    float2 acc[FH][FW];
#pragma unroll
    for (int fh = 0; fh < FH; ++fh)
#pragma unroll
        for (int fw = 0; fw < FW; ++fw) acc[fh][fw] = make_float2(0.f, 0.f);

    int v = z;
    if (tid == 0 && v < g.per_ctile) issue(v, 0);
    for (int k = 0; v < g.per_ctile; ++k, v += Zc) {
        const int vn = v + Zc;
        if (tid == 0 && vn < g.per_ctile) issue(vn, (k + 1) & 1);
        if (!mbar_wait(&bars[k & 1], (k >> 1) & 1)) {
            report_timeout(err);
            if (tid == 0 && vn < g.per_ctile) mbar_wait(&bars[(k + 1) & 1], ((k + 1) >> 1) & 1);
            return;
        }

        const unsigned char *cur = smem_raw + (k & 1) * stage;
        const T *sx = reinterpret_cast<const T *>(cur) + img_l * halo_elems;
        const T *sy = reinterpret_cast<const T *>(cur + align128(hb)) + img_l * otile_elems;
        const int r0 = rt * TH, j0 = ct * TW;
        using M = typename std::conditional<!HA && sizeof(T) == 2 && FH == DWCONV_W_FFMA2_FH, MacW<T>,
                                            Mac<T>>::type;
        typename M::V dyv[TH][TW];
#pragma unroll
        for (int th = 0; th < TH; ++th)
#pragma unroll
            for (int tw = 0; tw < TW; ++tw)
                dyv[th][tw] = M::load(sy + ((r0 + th) * tile_cols + j0 + tw) * 32 + 2 * cp);
        if constexpr (HA) {
            static_assert(std::is_same<T, __half>::value, "hybrid accumulation is for fp16 data");
            __half2 part_h[FH][FW];
#pragma unroll
            for (int fh = 0; fh < FH; ++fh)
#pragma unroll
                for (int fw = 0; fw < FW; ++fw) part_h[fh][fw] = __float2half2_rn(0.f);
#pragma unroll
            for (int r = 0; r < TH + FH - 1; ++r) {
                __half2 xv[WW];
                const T *srow = sx + ((r0 + r) * g.HW + j0) * 32 + 2 * cp;
#pragma unroll
                for (int j = 0; j < WW; ++j) xv[j] = *reinterpret_cast<const __half2 *>(srow + j * 32);
#pragma unroll
                for (int th = 0; th < TH; ++th) {
                    const int fh = r - th;
                    if (fh < 0 || fh >= FH) continue;
#pragma unroll
                    for (int fw = 0; fw < FW; ++fw)
#pragma unroll
                        for (int tw = 0; tw < TW; ++tw) {
                            const unsigned d = dyv[th][tw];
                            part_h[fh][fw] =
                                __hfma2(*reinterpret_cast<const __half2 *>(&d), xv[tw + fw], part_h[fh][fw]);
                        }
                }
            }
#pragma unroll
            for (int fh = 0; fh < FH; ++fh)
#pragma unroll
                for (int fw = 0; fw < FW; ++fw) {
                    const float2 f = __half22float2(part_h[fh][fw]);
                    acc[fh][fw].x += f.x;
                    acc[fh][fw].y += f.y;
                }
        } else {
#pragma unroll
            for (int r = 0; r < TH + FH - 1; ++r) {
                typename M::V xv[WW];
                const T *srow = sx + ((r0 + r) * g.HW + j0) * 32 + 2 * cp;
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
                            M::fma(acc[fh][fw], dyv[th][tw], xv[tw + fw]);
                }
            }
        }
        __syncthreads();  // this buffer is refilled by the copy issued next iteration
    }

    // Sum the 8 thread tiles that share each channel pair: lanes l and l^16 of a
    // warp hold tiles 2w and 2w+1; then the four warps, in a fixed order.
    float2 *red = reinterpret_cast<float2 *>(smem_raw);  // [4][FH*FW][16]
    const int warp = tid / 32, lane = tid % 32;
#pragma unroll
    for (int fh = 0; fh < FH; ++fh)
#pragma unroll
        for (int fw = 0; fw < FW; ++fw) {
            float2 a = acc[fh][fw];
            a.x += __shfl_xor_sync(0xffffffffu, a.x, 16);
            a.y += __shfl_xor_sync(0xffffffffu, a.y, 16);
            if (lane < 16) red[(warp * FH * FW + fh * FW + fw) * 16 + lane] = a;
        }
    __syncthreads();
    for (int idx = tid; idx < FH * FW * 16; idx += kThreads) {
        const int tap = idx / 16, pr = idx % 16;
        float2 s = red[tap * 16 + pr];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) {
            const float2 o = red[(w * FH * FW + tap) * 16 + pr];
            s.x += o.x;
            s.y += o.y;
        }
        const int c = ctile * 32 + 2 * pr;
        if (c < p.C) {
            float *dst = part + ((long long)z * FH * FW + tap) * p.C + c;
            dst[0] = s.x;
            dst[1] = s.y;
        }
    }
}

// Plan: which instance, its geometry, and the slice count Zc -- about one
// full wave: the SMs x the CTAs of this instance that fit on an SM (its
// register bound MINB, or fewer if shared memory holds fewer).  Planned for
// the bounds of plan_sms / plan_smem_per_sm (workspace size) or the current
// device (launch), so the launch's Zc never exceeds the workspace's.
template <typename T, int FH, int FW, int TH, int TW, int MINB>
bool plan_geo(const TiledConv &p, Geo &g, int &Zc, size_t &smem, bool launch) {
    g = make_geo(p, TH, TW, sizeof(T), true, sizeof(T) == 2 ? DWCONV_W16_SMEM_KB * 1024 : 110 * 1024);
    if (g.units == 0) return false;
    smem = stage_bytes(g, TH, TW, sizeof(T), true);
    const size_t red_bytes = (size_t)(kThreads / 32) * FH * FW * 16 * sizeof(float2);
    if (smem < red_bytes) smem = red_bytes;
    if (smem > 220 * 1024) return false;
    const int resident = std::max(1, std::min(MINB, (int)(plan_smem_per_sm(launch) / (smem + 1024))));
    int z = plan_sms(launch) * resident / g.ctiles;
    if (z > g.per_ctile) z = g.per_ctile;
    if (z < 1) z = 1;
    Zc = z;
    return true;
}

template <typename T, int FH, int FW, int TH, int TW, int MINB, bool HA = false>
cudaError_t run(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st) {
    Geo g;
    int Zc;
    size_t smem;
    if (!plan_geo<T, FH, FW, TH, TW, MINB>(p, g, Zc, smem, true)) return cudaErrorNotSupported;
    auto kern = tiled_wgrad_kernel<T, FH, FW, TH, TW, MINB, HA>;
    CUtensorMap halo_map, dy_map;
    if (!make_halo_map(&halo_map, p, g, dt, sizeof(T)) ||
        !make_tile_map(&dy_map, p.dy, p, g, TH, TW, dt, sizeof(T)))
        return cudaErrorNotSupported;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kThreads, smem, nullptr);
    if (e != cudaSuccess) return e;
    kern<<<g.ctiles * Zc, kThreads, smem, st>>>(halo_map, dy_map, p, g, part, Zc, device_error_word());
    note_launches(1);
    note_kernel(HA ? "tiled_wgrad_ha" : "tiled_wgrad");
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_wgrad_reduce(part, Zc, (long long)p.FH * p.FW * p.C, static_cast<float *>(p.out), st);
}

template <typename T>
cudaError_t dispatch(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st, int *Zc_out) {
    constexpr bool k16 = sizeof(T) == 2;
    constexpr int TH7 = k16 ? DWCONV_W16_TH : 4, TW7 = k16 ? DWCONV_W16_TW : 7;
    constexpr int MB7 = k16 ? DWCONV_W16_MINB : 2;
    Geo g;
    size_t smem;
    int Zc = 0;
    bool ok = false;
    const bool launch = Zc_out == nullptr;
    if (p.FH == 7 && p.FW == 7) ok = plan_geo<T, 7, 7, TH7, TW7, MB7>(p, g, Zc, smem, launch);
    else if (p.FH == 5 && p.FW == 5) ok = plan_geo<T, 5, 5, 4, 7, 2>(p, g, Zc, smem, launch);
    else if (p.FH == 3 && p.FW == 3) ok = plan_geo<T, 3, 3, 4, 7, 3>(p, g, Zc, smem, launch);
    if (!ok) return cudaErrorNotSupported;
    if (Zc_out) {  // planning only
        *Zc_out = Zc;
        return cudaSuccess;
    }
    if constexpr (std::is_same<T, __half>::value) {
        if (p.half_accumulate) {
            if (p.FH == 7) return run<T, 7, 7, TH7, TW7, DWCONV_WHA_MINB, true>(p, dt, part, st);
            if (p.FH == 5) return run<T, 5, 5, 4, 7, 2, true>(p, dt, part, st);
            return run<T, 3, 3, 4, 7, 3, true>(p, dt, part, st);
        }
    }
    if (p.FH == 7) return run<T, 7, 7, TH7, TW7, MB7>(p, dt, part, st);
    if (p.FH == 5) return run<T, 5, 5, 4, 7, 2>(p, dt, part, st);
    return run<T, 3, 3, 4, 7, 3>(p, dt, part, st);
}

template <typename F>
cudaError_t by_dtype(dwconv_dtype dt, F &&f) {
    switch (dt) {
        case DWCONV_FP32: return f(float{});
        case DWCONV_FP16: return f(__half{});
        case DWCONV_BF16: return f(__nv_bfloat16{});
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

int tiled_wgrad_slices(const TiledConv &p, dwconv_dtype dt) {
    int Zc = 0;
    cudaError_t e = by_dtype(dt, [&](auto tag) {
        return dispatch<decltype(tag)>(p, dt, nullptr, nullptr, &Zc);
    });
    return e == cudaSuccess ? Zc : 0;
}

cudaError_t launch_tiled_wgrad(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st) {
    return by_dtype(dt, [&](auto tag) { return dispatch<decltype(tag)>(p, dt, part, st, nullptr); });
}

}  // namespace dwc
