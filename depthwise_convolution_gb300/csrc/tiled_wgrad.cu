// Register-tiled weight gradient for small filters (Flash-DWC §5.1, "BFC").
//
//   dw[fh,fw,c] = sum over (n, i, j) of dy[n,i,j,c] * x_sub[n, i - pad + fh, j - pad + fw, c]
//
// on the same sub-grid description as the forward pass (tiled_common.cuh).
// The output dw is tiny (FH*FW*C) while the accumulation axis N*OH*OW is
// long, so the work is split along the accumulation axis (§5.1
// "accumulation-axis parallelisation"):
//   * grid = channel tiles x Zc; CTA (ctile, z) takes the work units
//     z, z + Zc, z + 2 Zc, ... of its channel tile, staging each unit's x halo
//     and dy tile in shared memory with cp.async (double-buffered);
//   * every thread keeps the FH x FW fp32 accumulators of its channel pair in
//     registers for the whole CTA, and walks its window row-stationary: each
//     x row is read once and feeds every (dy row, filter row) pair using it;
//     each multiply-add is a packed fma.rn.f32x2;
//   * at the end the 8 thread tiles sharing a channel pair are summed with a
//     warp shuffle and a fixed-order pass through shared memory, and the CTA
//     writes part[z][fh*FW+fw][c];
//   * wgrad_reduce (direct.cu) then sums the Zc slices in a fixed order, so
//     the result is bit-identical from call to call (no atomics).
#include "tiled_common.cuh"

namespace dwc {
namespace {

using namespace tiled;

constexpr int kTargetCtas = 304;  // two CTAs on each of the 152 SMs of a GB300

template <typename T, int FH, int FW, int TH, int TW, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    tiled_wgrad_kernel(TiledConv p, Geo g, float *__restrict__ part, int Zc) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
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
    const int stage_elems = g.NI * (halo_elems + otile_elems);
    T *st0 = reinterpret_cast<T *>(smem_raw);
    T *st1 = st0 + stage_elems;
    const T *dy = static_cast<const T *>(p.dy);

    const int ctile = blockIdx.x / Zc;
    const int z = blockIdx.x % Zc;
    const long long base = (long long)ctile * g.per_ctile;

    float2 acc[FH][FW];
#pragma unroll
    for (int fh = 0; fh < FH; ++fh)
#pragma unroll
        for (int fw = 0; fw < FW; ++fw) acc[fh][fw] = make_float2(0.f, 0.f);

    long long v = z;
    if (v < g.per_ctile) {
        {
            const Unit u0 = decode(g, base + v);
            stage_halo<T, TH, TW>(p, g, st0, u0);
            stage_out_tile<T, TH, TW>(p, g, dy, st0 + g.NI * halo_elems, u0);
        }
        cp_async_commit();
        for (int k = 0; v < g.per_ctile; ++k, v += Zc) {
            const long long vn = v + Zc;
            if (vn < g.per_ctile) {
                T *nb = (k & 1) ? st0 : st1;
                const Unit un = decode(g, base + vn);
                stage_halo<T, TH, TW>(p, g, nb, un);
                stage_out_tile<T, TH, TW>(p, g, dy, nb + g.NI * halo_elems, un);
            }
            cp_async_commit();
            cp_async_wait_1();
            __syncthreads();

            const T *buf = (k & 1) ? st1 : st0;
            const T *sx = buf + (long long)img_l * halo_elems;
            const T *sy = buf + (long long)g.NI * halo_elems + (long long)img_l * otile_elems;
            const int r0 = rt * TH, j0 = ct * TW;
            float2 dyv[TH][TW];
#pragma unroll
            for (int th = 0; th < TH; ++th)
#pragma unroll
                for (int tw = 0; tw < TW; ++tw)
                    dyv[th][tw] = Pair<T>::load(sy + ((long long)(r0 + th) * tile_cols + j0 + tw) * 32 + 2 * cp);
#pragma unroll
            for (int r = 0; r < TH + FH - 1; ++r) {
                float2 xv[WW];
                const T *srow = sx + ((long long)(r0 + r) * g.HW + j0) * 32 + 2 * cp;
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
                            acc[fh][fw] = __ffma2_rn(dyv[th][tw], xv[tw + fw], acc[fh][fw]);
                }
            }
            __syncthreads();  // this buffer is restaged two units from now
        }
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

// Shape-only plan: which instance, its geometry, and the slice count Zc.
template <typename T, int FH, int FW, int TH, int TW>
bool plan_geo(const TiledConv &p, Geo &g, int &Zc, size_t &smem) {
    g = make_geo(p, TH, TW, sizeof(T), true, 110 * 1024);
    smem = stage_bytes(g, TH, TW, sizeof(T), true);
    const size_t red_bytes = (size_t)(kThreads / 32) * FH * FW * 16 * sizeof(float2);
    if (smem < red_bytes) smem = red_bytes;
    if (smem > 220 * 1024) return false;
    long long z = kTargetCtas / g.ctiles;
    if (z > g.per_ctile) z = g.per_ctile;
    if (z < 1) z = 1;
    Zc = (int)z;
    return true;
}

template <typename T, int FH, int FW, int TH, int TW, int MINB>
cudaError_t run(const TiledConv &p, float *part, cudaStream_t st) {
    Geo g;
    int Zc;
    size_t smem;
    if (!plan_geo<T, FH, FW, TH, TW>(p, g, Zc, smem)) return cudaErrorNotSupported;
    auto kern = tiled_wgrad_kernel<T, FH, FW, TH, TW, MINB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<g.ctiles * Zc, kThreads, smem, st>>>(p, g, part, Zc);
    note_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_wgrad_reduce(part, Zc, (long long)p.FH * p.FW * p.C, static_cast<float *>(p.out), st);
}

template <typename T>
cudaError_t dispatch(const TiledConv &p, float *part, cudaStream_t st, int *Zc_out) {
    Geo g;
    size_t smem;
    int Zc = 0;
    bool ok = false;
    if (p.FH == 7 && p.FW == 7) ok = plan_geo<T, 7, 7, 4, 7>(p, g, Zc, smem);
    else if (p.FH == 5 && p.FW == 5) ok = plan_geo<T, 5, 5, 4, 7>(p, g, Zc, smem);
    else if (p.FH == 3 && p.FW == 3) ok = plan_geo<T, 3, 3, 4, 7>(p, g, Zc, smem);
    if (!ok) return cudaErrorNotSupported;
    if (Zc_out) {  // planning only
        *Zc_out = Zc;
        return cudaSuccess;
    }
    if (p.FH == 7) return run<T, 7, 7, 4, 7, 2>(p, part, st);
    if (p.FH == 5) return run<T, 5, 5, 4, 7, 2>(p, part, st);
    return run<T, 3, 3, 4, 7, 3>(p, part, st);
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
        return dispatch<decltype(tag)>(p, nullptr, nullptr, &Zc);
    });
    return e == cudaSuccess ? Zc : 0;
}

cudaError_t launch_tiled_wgrad(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st) {
    return by_dtype(dt, [&](auto tag) { return dispatch<decltype(tag)>(p, part, st, nullptr); });
}

}  // namespace dwc
