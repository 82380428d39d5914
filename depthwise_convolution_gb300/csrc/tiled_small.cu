// Register-tiled forward pass and input gradient for small filters (3x3, 5x5, 7x7).
//
// Design (the Flash-DWC §3.1-§3.4 dataflow restated for sm_103a):
//   * Work units, CTA shape and halo staging: see tiled_common.cuh.  Two
//     stage buffers: the next unit's halo streams in while this one computes.
//   * The channel pair's FH x FW filter lives in registers as fp32 pairs and
//     is reloaded only when the channel tile changes (filter reuse across all
//     spatial positions a thread computes, §3.2).
//   * Width-first register reuse (§3.3): the thread walks the TH+FH-1 input
//     rows of its window once; each row's TW+FW-1 values are read from shared
//     memory once, widened to fp32 once, and feed every (output row, filter
//     row) pair that uses that input row.  Each multiply-add is a packed
//     fma.rn.f32x2 over the channel pair, accumulating in fp32.
//   * Persistent grid: as many CTAs as fit on the SMs, each taking work units
//     round-robin, so the last wave is at most one unit deep.
//   * Epilogue: bias added once (forward only), round to the storage type,
//     masked stores for spatial and channel tails; with zero_phases the other
//     output phases of each stride block are written as zeros.
#include "tiled_common.cuh"

namespace dwc {
namespace {

using namespace tiled;

template <typename T, int FH, int FW, int TH, int TW, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) tiled_small_kernel(TiledConv p, Geo g) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int WW = TW + FW - 1;  // input columns one thread reads per row

    const int tid = threadIdx.x;
    const int cp = tid % kPairs;
    const int t = tid / kPairs;
    const int img_l = t / (g.RT * g.CT);
    const int rt = (t / g.CT) % g.RT;
    const int ct = t % g.CT;

    const int halo_elems = g.HH * g.HW * 32;
    T *sbuf0 = reinterpret_cast<T *>(smem_raw);
    T *sbuf1 = sbuf0 + g.NI * halo_elems;
    const T *wgt = static_cast<const T *>(p.w);
    T *out = static_cast<T *>(p.out);
    const int tile_rows = g.RT * TH, tile_cols = g.CT * TW;

    float2 wr[FH][FW];
    float2 bias2 = make_float2(0.f, 0.f);
    int loaded_ctile = -1;

    long long u = blockIdx.x;
    if (u >= g.units) return;
    stage_halo<T, TH, TW>(p, g, sbuf0, decode(g, u));
    cp_async_commit();
    for (int k = 0; u < g.units; ++k, u += gridDim.x) {
        const long long un = u + gridDim.x;
        if (un < g.units) stage_halo<T, TH, TW>(p, g, (k & 1) ? sbuf0 : sbuf1, decode(g, un));
        cp_async_commit();
        cp_async_wait_1();
        __syncthreads();

        const Unit cur = decode(g, u);
        const int c = cur.ctile * 32 + 2 * cp;
        const bool cvalid = c < p.C;
        if (cur.ctile != loaded_ctile) {
            loaded_ctile = cur.ctile;
#pragma unroll
            for (int fh = 0; fh < FH; ++fh)
#pragma unroll
                for (int fw = 0; fw < FW; ++fw) {
                    const int sfh = p.flip ? FH - 1 - fh : fh;
                    const int sfw = p.flip ? FW - 1 - fw : fw;
                    wr[fh][fw] = cvalid ? Pair<T>::load(wgt + ((long long)sfh * FW + sfw) * p.C + c)
                                        : make_float2(0.f, 0.f);
                }
            bias2 = (p.bias && cvalid) ? make_float2(p.bias[c], p.bias[c + 1]) : make_float2(0.f, 0.f);
        }

        const T *s = ((k & 1) ? sbuf1 : sbuf0) + (long long)img_l * halo_elems;
        const int r0 = rt * TH, j0 = ct * TW;
        float2 acc[TH][TW];
#pragma unroll
        for (int th = 0; th < TH; ++th)
#pragma unroll
            for (int tw = 0; tw < TW; ++tw) acc[th][tw] = bias2;

#pragma unroll
        for (int r = 0; r < TH + FH - 1; ++r) {
            float2 xv[WW];
            const T *srow = s + ((long long)(r0 + r) * g.HW + j0) * 32 + 2 * cp;
#pragma unroll
            for (int j = 0; j < WW; ++j) xv[j] = Pair<T>::load(srow + j * 32);
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int fh = r - th;
                if (fh < 0 || fh >= FH) continue;
#pragma unroll
                for (int fw = 0; fw < FW; ++fw)
#pragma unroll
                    for (int tw = 0; tw < TW; ++tw)
                        acc[th][tw] = __ffma2_rn(wr[fh][fw], xv[tw + fw], acc[th][tw]);
            }
        }

        const int n = cur.group * g.NI + img_l;
        if (cvalid && n < p.N) {
            const int i0 = cur.band * tile_rows + r0;
            const int jj0 = cur.twi * tile_cols + j0;
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int i = i0 + th;
                if (i >= p.OHs) break;
#pragma unroll
                for (int tw = 0; tw < TW; ++tw) {
                    const int j = jj0 + tw;
                    if (j >= p.OWs) break;
                    const int orow = p.out_off + p.out_step * i;
                    const int ocol = p.out_off + p.out_step * j;
                    if (orow < p.OHf && ocol < p.OWf)
                        Pair<T>::store(out + (((long long)n * p.OHf + orow) * p.OWf + ocol) * p.C + c,
                                       acc[th][tw]);
                    if (p.zero_phases) {
                        for (int a = 0; a < p.out_step; ++a)
                            for (int b = 0; b < p.out_step; ++b) {
                                if (a == p.out_off && b == p.out_off) continue;
                                const int zr = p.out_step * i + a, zc = p.out_step * j + b;
                                if (zr < p.OHf && zc < p.OWf)
                                    Pair<T>::store(out + (((long long)n * p.OHf + zr) * p.OWf + zc) * p.C + c,
                                                   make_float2(0.f, 0.f));
                            }
                    }
                }
            }
        }
        __syncthreads();  // this buffer is restaged two units from now
    }
}

template <typename T, int FH, int FW, int TH, int TW, int MINB>
cudaError_t run(const TiledConv &p, cudaStream_t st) {
    auto kern = tiled_small_kernel<T, FH, FW, TH, TW, MINB>;
    const Geo g = make_geo(p, TH, TW, sizeof(T), false, 100 * 1024);
    const size_t smem = stage_bytes(g, TH, TW, sizeof(T), false);
    if (smem > 220 * 1024) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const long long slots = (long long)sm_count() * per_sm;
    const int grid = (int)std::min<long long>(g.units, slots);
    kern<<<grid, kThreads, smem, st>>>(p, g);
    note_launches(1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_filter(const TiledConv &p, cudaStream_t st) {
    if (p.FH == 7 && p.FW == 7) return run<T, 7, 7, 4, 7, 2>(p, st);
    if (p.FH == 5 && p.FW == 5) return run<T, 5, 5, 4, 7, 2>(p, st);
    if (p.FH == 3 && p.FW == 3) return run<T, 3, 3, 4, 7, 3>(p, st);
    if (p.FH == 3 && p.FW == 5) return run<T, 3, 5, 4, 7, 3>(p, st);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_tiled_small(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    switch (dt) {
        case DWCONV_FP32: return dispatch_filter<float>(p, st);
        case DWCONV_FP16: return dispatch_filter<__half>(p, st);
        case DWCONV_BF16: return dispatch_filter<__nv_bfloat16>(p, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
