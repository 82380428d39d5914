// Register-tiled depthwise convolution for small filters (3x3, 5x5, 7x7).
//
// Design (restating Flash-DWC §3.1-§3.4 for sm_103a; see the notes below for
// what differs from the paper's A100/RTX 4090 kernel):
//   * Work unit = one output tile of (NI images) x (RT*TH rows) x (CT*TW
//     columns) x 32 channels.  The CTA is 16 channel pairs x 8 thread tiles
//     (NI*RT*CT = 8), 128 threads; every thread owns one channel pair and a
//     TH x TW block of outputs.
//   * The input halo of a tile, (RT*TH-1)+FH rows by (CT*TW-1)+FW columns
//     ("Tiles, halos and partial sums": (T-1)S + (R-1)D + 1 with S = D = 1 on
//     the sub-grid), is staged in shared memory with 16-byte cp.async copies.
//     Copies that fall outside the input use a zero source size, so the
//     padding is generated as zeros in shared memory rather than fetched.
//     Two buffers: the next unit's halo streams in while this one computes.
//   * The channel pair's FH x FW filter lives in registers as fp32 pairs and
//     is reloaded only when the channel tile changes (filter reuse across all
//     spatial positions a thread computes, §3.2).
//   * Width-first register reuse (§3.3): the thread walks the TH+FH-1 input
//     rows of its window once; each row's TW+FW-1 values are loaded into
//     registers once, widened to fp32 once, and feed every (output row,
//     filter row) pair that uses that input row.  Each FMA is a packed
//     fma.rn.f32x2 over the channel pair, accumulating in fp32.
//   * Persistent grid: as many CTAs as fit on the SMs, each taking work units
//     round-robin, so the last wave is at most one unit deep.
//   * Epilogue: bias added once (forward only), round to the storage type,
//     masked stores for spatial and channel tails (§"Tiles, halos and
//     partial sums": mask the final spatial and channel tiles).
#include <algorithm>

#include "common.cuh"

namespace dwc {
namespace {

constexpr int kPairs = 16;                 // channel pairs per CTA (32 channels)
constexpr int kTiles = 8;                  // thread tiles per CTA
constexpr int kThreads = kPairs * kTiles;  // 128

struct Geo {
    int NI, RT, CT;        // thread tiles: images x rows x columns (product 8)
    int HH, HW;            // halo rows / columns per image
    int tiles_h, tiles_w;  // work units along output rows / columns
    int groups, ctiles;    // image groups (NI images each), channel tiles
    long long units;       // ctiles * groups * tiles_w * tiles_h
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

template <typename T, int FH, int FW, int TH, int TW, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) tiled_small_kernel(TiledConv p, Geo g) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int EPC = 16 / sizeof(T);  // elements per 16-byte copy
    constexpr int CPP = 32 / EPC;        // copies per pixel (32 channels)
    constexpr int WW = TW + FW - 1;      // input columns one thread reads per row

    const int tid = threadIdx.x;
    const int cp = tid % kPairs;
    const int t = tid / kPairs;
    const int img_l = t / (g.RT * g.CT);
    const int rt = (t / g.CT) % g.RT;
    const int ct = t % g.CT;

    const int halo_elems = g.HH * g.HW * 32;
    const int buf_elems = g.NI * halo_elems;
    T *sbuf0 = reinterpret_cast<T *>(smem_raw);
    T *sbuf1 = sbuf0 + buf_elems;
    const T *in = static_cast<const T *>(p.in);
    const T *wgt = static_cast<const T *>(p.w);
    T *out = static_cast<T *>(p.out);

    const int tile_rows = g.RT * TH, tile_cols = g.CT * TW;
    const long long per_ctile = (long long)g.groups * g.tiles_w * g.tiles_h;

    auto decode = [&](long long u, int &ctile, int &group, int &twi, int &band) {
        ctile = (int)(u / per_ctile);
        long long r = u % per_ctile;
        band = (int)(r % g.tiles_h);
        r /= g.tiles_h;
        twi = (int)(r % g.tiles_w);
        group = (int)(r / g.tiles_w);
    };

    auto stage = [&](T *dst, long long u) {
        int ctile, group, twi, band;
        decode(u, ctile, group, twi, band);
        const int ih0 = band * tile_rows - p.pad_h;
        const int iw0 = twi * tile_cols - p.pad_w;
        const int c0 = ctile * 32;
        const int total = g.NI * g.HH * g.HW * CPP;
        for (int k = tid; k < total; k += kThreads) {
            const int q = k % CPP;
            const int pix = k / CPP;
            const int b = pix % g.HW;
            const int a = (pix / g.HW) % g.HH;
            const int il = pix / (g.HW * g.HH);
            const int nn = group * g.NI + il;
            const int ihs = ih0 + a, iws = iw0 + b, cc = c0 + q * EPC;
            const bool ok = nn < p.N && ihs >= 0 && ihs < p.Hs && iws >= 0 && iws < p.Ws && cc < p.C;
            const T *src = in;
            if (ok)
                src += (((long long)nn * p.Hf + (p.in_off + p.in_step * ihs)) * p.Wf +
                        (p.in_off + p.in_step * iws)) * (long long)p.C + cc;
            cp_async16(dst + (long long)pix * 32 + q * EPC, src, ok ? 16 : 0);
        }
    };

    float2 wr[FH][FW];
    float2 bias2 = make_float2(0.f, 0.f);
    int loaded_ctile = -1;

    long long u = blockIdx.x;
    if (u >= g.units) return;
    stage(sbuf0, u);
    cp_async_commit();
    for (int k = 0; u < g.units; ++k, u += gridDim.x) {
        const long long un = u + gridDim.x;
        if (un < g.units) stage((k & 1) ? sbuf0 : sbuf1, un);
        cp_async_commit();
        cp_async_wait_1();
        __syncthreads();

        int ctile, group, twi, band;
        decode(u, ctile, group, twi, band);
        const int c = ctile * 32 + 2 * cp;
        const bool cvalid = c < p.C;
        if (ctile != loaded_ctile) {
            loaded_ctile = ctile;
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

        const int n = group * g.NI + img_l;
        if (cvalid && n < p.N) {
            const int i0 = band * tile_rows + r0;
            const int jj0 = twi * tile_cols + j0;
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

// ---- host side ---------------------------------------------------------------

int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Shape of the thread-tile grid for an OHs x OWs output: columns first, then
// rows, then images, so that a CTA's 8 thread tiles are all useful on small maps.
Geo make_geo(const TiledConv &p, int TH, int TW, size_t elem) {
    Geo g{};
    g.CT = std::min(8, next_pow2((p.OWs + TW - 1) / TW));
    g.RT = std::min(8 / g.CT, next_pow2((p.OHs + TH - 1) / TH));
    g.NI = 8 / (g.CT * g.RT);
    // keep the double-buffered halo within ~100 KB so two CTAs share an SM
    auto smem = [&](const Geo &q) {
        return 2 * (size_t)q.NI * (q.RT * TH + p.FH - 1) * (q.CT * TW + p.FW - 1) * 32 * elem;
    };
    while (smem(g) > 100 * 1024 && g.CT > 1) {
        g.CT /= 2;
        g.RT = std::min(8 / g.CT, next_pow2((p.OHs + TH - 1) / TH));
        g.NI = 8 / (g.CT * g.RT);
    }
    g.HH = g.RT * TH + p.FH - 1;
    g.HW = g.CT * TW + p.FW - 1;
    g.tiles_h = (p.OHs + g.RT * TH - 1) / (g.RT * TH);
    g.tiles_w = (p.OWs + g.CT * TW - 1) / (g.CT * TW);
    g.groups = (p.N + g.NI - 1) / g.NI;
    g.ctiles = (p.C + 31) / 32;
    g.units = (long long)g.ctiles * g.groups * g.tiles_w * g.tiles_h;
    return g;
}

template <typename T, int FH, int FW, int TH, int TW, int MINB>
cudaError_t run(const TiledConv &p, cudaStream_t st) {
    auto kern = tiled_small_kernel<T, FH, FW, TH, TW, MINB>;
    const Geo g = make_geo(p, TH, TW, sizeof(T));
    const size_t smem = 2 * (size_t)g.NI * g.HH * g.HW * 32 * sizeof(T);
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
