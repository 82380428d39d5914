// Tensor-core weight gradient for large 16-bit filters (FW >= 8 in the
// kernel's view; strips taller than wide arrive transposed).
//
//   dw[fh,fw,c] = sum over (n, i, j) of dy[n,i,j,c] * x_sub[n, i - pad_h + fh, j - pad_w + fw, c]
//
// For one channel, one dy row i and the x row i + fh, the sum over j is a 1-D
// correlation; over a tile it becomes a GEMM whose A operand is a Toeplitz
// band of dy (the Flash-DWC §4.2 packing with dy in the filter's place):
//
//   D[m][n] += sum_{k<16} A[m][k] B[k][n],  A[m][k] = dy[i][J0 + k - fw(m)],  B[k][n] = x[i + fh(n)][J0 + k],
//
// an mma.sync m16n8k16 (16-bit in, fp32 accumulate) per 16 x columns J0, 16
// filter columns fw(m) = 16 fb + m and 8 filter rows fh(n) = 8 hb + n.  Every
// x column meets every dy column exactly once, so no band is masked: dy
// outside the tile is zero in the staged copy.
//
// Work unit: 8 channels (one per warp) x OTH dy rows x OTW dy columns of one
// image, 256 threads.  Per unit one thread stages the x halo the taps read and
// the dy tile with two TMA copies on one mbarrier (double-buffered, bounded
// waits); ldmatrix.trans + stmatrix build channel-major copies of both (dy
// twice, the second shifted by one column, so that every A pair is one
// aligned 32-bit load); each warp then runs its channel's MMAs with the
// NFB x NHB accumulator blocks in registers for the whole CTA.  Grid =
// channel tiles x accumulation slices; each CTA writes its slice of the
// partial sums and wgrad_reduce (direct.cu) sums the slices in a fixed order.
#include "mma_common.cuh"

namespace dwc {
namespace {

using namespace tiled;
using namespace mma;

constexpr int kWCh = 8;            // channels per unit, one per warp
constexpr int kWThreads = 256;
#ifndef DWCONV_WG_OTH
#define DWCONV_WG_OTH 4
#endif
#ifndef DWCONV_WG_OTW
#define DWCONV_WG_OTW 64
#endif
// dy rows, columns per unit (measured on GB300: 4 x 64 beats 8 x 32 by 8-15 %,
// the wider tile wasting fewer Toeplitz products at its edges)
constexpr int kWOTH = DWCONV_WG_OTH, kWOTW = DWCONV_WG_OTW;

template <int NFB, int NHB>
struct CfgW {
    static constexpr int FWMAX = 16 * NFB, FHMAX = 8 * NHB;
    // x halo: rows OTH + FH - 1 staged, OTH + 8 NHB - 1 allocated (the last
    // block's surplus rows only reach unused accumulator columns); columns
    // OTW + FW - 1 rounded up to whole 16-column groups, NG of them at most.
    static constexpr int NG = (kWOTW + FWMAX - 1 + 15) / 16;
    static constexpr int SWX = 16 * NG;
    static constexpr int TXR = kWOTH + FHMAX - 1;
    // T_x row stride: 8 rows of a B load fall in distinct bank quads.
    static constexpr int RSX = SWX % 16 == 8 ? SWX : SWX + ((8 - SWX % 16 + 16) % 16);
    static constexpr int CSX = TXR * RSX;
    // T_dy: dy column e sits at LM + e; A reads e from -(16 NFB - 1) to 16 NG.
    static constexpr int LM = 16 * NFB;
    static constexpr int DW = LM + SWX + 8;
    static constexpr int CSD = 2 * kWOTH * DW + 16;  // two copies; +16 halves: copies apart in banks
    static constexpr unsigned x_bytes_max = (unsigned)(kWOTH + FHMAX - 1) * SWX * 16;
    static constexpr unsigned dy_bytes = kWOTH * kWOTW * 16;
    static constexpr unsigned dy_off = align1k(x_bytes_max);  // dy box within a stage
    static constexpr unsigned stage = dy_off + align1k(dy_bytes);
    static constexpr unsigned tx_off = 2 * stage;
    static constexpr unsigned td_off = tx_off + align1k(kWCh * CSX * 2);
    static constexpr unsigned zero_off = td_off + align1k(kWCh * CSD * 2);
    static constexpr unsigned smem = zero_off + 16;
};

struct GeoWM {
    int tiles_h, tiles_w, per_ctile, ctiles;
    int HR;            // x halo rows staged (OTH + FH - 1)
    unsigned x_bytes;  // bytes of the staged x box
};

template <typename T, int NFB, int NHB>
__global__ void __launch_bounds__(kWThreads, 2)
    tiled_mma_wgrad_kernel(const __grid_constant__ CUtensorMap halo_map, const __grid_constant__ CUtensorMap dy_map,
                           TiledConv p, GeoWM g, float *__restrict__ part, int Zc, unsigned *err) {
    using C = CfgW<NFB, NHB>;
    constexpr int NG = C::NG;
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    __shared__ __align__(8) uint64_t bars[2];

    unsigned char *smem_raw = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int gq = lane / 4, t4 = lane % 4;
    const int tr = lane % 8, tj = lane / 8;
    const unsigned s_addr = smem_addr(smem_raw);
    const unsigned tx_addr = s_addr + C::tx_off, td_addr = s_addr + C::td_off, zero_addr = s_addr + C::zero_off;
    const int ctile = blockIdx.x / Zc, z = blockIdx.x % Zc;

    // Zero T_x and T_dy once: margins and surplus rows are never written again.
    for (unsigned i = tid; i < (C::zero_off + 16 - C::tx_off) / 16; i += kWThreads)
        reinterpret_cast<uint4 *>(smem_raw + C::tx_off)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    auto issue = [&](int v, int b) {
        const int band = v % g.tiles_h, rest = v / g.tiles_h;
        const int twi = rest % g.tiles_w, n = rest / g.tiles_w;
        unsigned char *dst = smem_raw + b * C::stage;
        mbar_arrive_expect_tx(&bars[b], g.x_bytes + C::dy_bytes);
        tma_load_4d(dst, &halo_map, ctile * kWCh, twi * kWOTW - p.pad_w, band * kWOTH - p.pad_h, n, &bars[b]);
        tma_load_4d(dst + C::dy_off, &dy_map, ctile * kWCh, twi * kWOTW, band * kWOTH, n, &bars[b]);
    };

    float acc[NFB][NHB][4];
#pragma unroll
    for (int fb = 0; fb < NFB; ++fb)
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) acc[fb][hb][0] = acc[fb][hb][1] = acc[fb][hb][2] = acc[fb][hb][3] = 0.f;

    // This warp's channel in T_x / T_dy (halves).
    const unsigned tx_c = tx_addr + 2u * (unsigned)(warp * C::CSX);
    const unsigned td_c = td_addr + 2u * (unsigned)(warp * C::CSD);
    // A pair of lane (gq, t4), block fb, group grp: dy columns e, e+1 with
    // e = 8 grp + 2t4 - 16 fb - gq (- 8 for M rows 8-15); copy q = gq & 1
    // holds dy[e'] at column LM + e' + q, where e + q is even.
    const int q = gq & 1;
    const unsigned a_lane = td_c + 2u * (unsigned)(q * kWOTH * C::DW + C::LM + 2 * t4 - gq + q);
    // B pair: x row i + 8 hb + gq, columns 8 grp + 2t4, +1.
    const unsigned b_lane = tx_c + 2u * (unsigned)(gq * C::RSX + 2 * t4);

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
        const unsigned sx = s_addr + (k & 1) * C::stage;
        const unsigned sd = sx + C::dy_off;
        // Transpose the x halo [HR][SWX][8 ch] -> T_x[ch][row][col], four
        // 8-pixel blocks per step (lane (tr, tj) addresses pixel tr of block
        // tj); blocks past the last repeat it (same data to the same place).
        {
            constexpr int CB = C::SWX / 8;  // 8-pixel blocks per row
            const int nb = g.HR * CB;
            for (int m0 = warp * 4; m0 < nb; m0 += kWThreads / 8) {
                const int m = min(m0 + tj, nb - 1);
                const int row = m / CB, col0 = (m % CB) * 8;
                unsigned v0, v1, v2, v3;
                ldsm_x4_trans(v0, v1, v2, v3, sx + (unsigned)((row * C::SWX + col0 + tr) * 16));
                stsm_x4(tx_addr + 2u * (unsigned)(tr * C::CSX + row * C::RSX + col0), v0, v1, v2, v3);
            }
        }
        // dy: copy 0 at columns LM + j, copy 1 (dy[j - 1]) at LM + j; copy 1's
        // blocks start one pixel early, with the zero pixel outside the tile.
        {
            constexpr int nb0 = kWOTH * (kWOTW / 8), nb1 = kWOTH * (kWOTW / 8 + 1);
            for (int m0 = warp * 4; m0 < nb0 + nb1; m0 += kWThreads / 8) {
                const int m = min(m0 + tj, nb0 + nb1 - 1);
                const bool shifted = m >= nb0;
                const int mm = shifted ? m - nb0 : m;
                const int per = shifted ? kWOTW / 8 + 1 : kWOTW / 8;
                const int row = mm / per, col0 = (mm % per) * 8;
                const int px = col0 + tr - (shifted ? 1 : 0);
                const unsigned src =
                    (px >= 0 && px < kWOTW) ? sd + (unsigned)((row * kWOTW + px) * 16) : zero_addr;
                unsigned v0, v1, v2, v3;
                ldsm_x4_trans(v0, v1, v2, v3, src);
                stsm_x4(td_addr + 2u * (unsigned)(tr * C::CSD + (shifted ? kWOTH * C::DW : 0) + row * C::DW +
                                                  C::LM + col0),
                        v0, v1, v2, v3);
            }
        }
        __syncthreads();  // T_x, T_dy ready; this staging buffer is free

        // MMAs of this warp's channel, 16 x columns each (m16n8k16).  A of
        // block fb, group grp holds dy columns e0 = 16 grp + 2t4 - 16 fb - gq
        // (a0), e0 - 8 (a1, M rows 8-15), e0 + 8 (a2, k 8-15) and e0 again
        // (a3: rows 8-15 and k 8-15 cancel).  Blocks (grp, fb) whose x columns
        // meet no dy column of the tile are skipped at compile time.
#pragma unroll 1
        for (int i = 0; i < kWOTH; ++i) {
#pragma unroll
            for (int grp = 0; grp < NG; ++grp) {
                unsigned b[NHB][2];
#pragma unroll
                for (int hb = 0; hb < NHB; ++hb) {
                    const unsigned ba = b_lane + 2u * (unsigned)((i + 8 * hb) * C::RSX + 16 * grp);
                    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(b[hb][0]) : "r"(ba));
                    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(b[hb][1]) : "r"(ba + 16u));
                }
#pragma unroll
                for (int fb = 0; fb < NFB; ++fb) {
                    // dy columns 16 grp - 16 fb - 15 .. 16 grp - 16 fb + 15.
                    if (16 * grp - 16 * fb + 15 < 0 || 16 * grp - 16 * fb - 15 >= kWOTW) continue;
                    const unsigned a = a_lane + 2u * (unsigned)(i * C::DW + 16 * grp - 16 * fb);
                    unsigned a0, a1, a2;
                    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(a0) : "r"(a));
                    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(a1) : "r"(a - 16u));  // 8 columns left
                    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(a2) : "r"(a + 16u));  // 8 columns right
#pragma unroll
                    for (int hb = 0; hb < NHB; ++hb) MmaOp<T>::run(acc[fb][hb], a0, a1, a2, a0, b[hb][0], b[hb][1]);
                }
            }
        }
        __syncthreads();  // every warp is done with T_x / T_dy
    }

    // D[m][n] of block (fb, hb): lane (gq, t4) holds m = gq (+8), n = 2t4 (+1).
    const int c = ctile * kWCh + warp;
    if (c >= p.C) return;
#pragma unroll
    for (int fb = 0; fb < NFB; ++fb)
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int fw = 16 * fb + gq + 8 * (r >> 1), fh = 8 * hb + 2 * t4 + (r & 1);
                if (fw >= p.FW || fh >= p.FH) continue;
                const int tap = p.transpose ? fw * p.FH + fh : fh * p.FW + fw;  // memory order
                part[((long long)z * p.FH * p.FW + tap) * p.C + c] = acc[fb][hb][r];
            }
}

// Compiled accumulator shapes (filter column blocks of 16 x row blocks of 8),
// smallest first; the first that covers the filter is taken.
template <typename F>
cudaError_t with_shape(int FH, int FW, F &&f) {
    const int nfb = (FW + 15) / 16, nhb = (FH + 7) / 8;
    if (nfb <= 1 && nhb <= 1) return f(std::integral_constant<int, 1>{}, std::integral_constant<int, 1>{});
    if (nfb <= 1 && nhb <= 2) return f(std::integral_constant<int, 1>{}, std::integral_constant<int, 2>{});
    if (nfb <= 2 && nhb <= 1) return f(std::integral_constant<int, 2>{}, std::integral_constant<int, 1>{});
    if (nfb <= 2 && nhb <= 2) return f(std::integral_constant<int, 2>{}, std::integral_constant<int, 2>{});
    if (nfb <= 2 && nhb <= 3) return f(std::integral_constant<int, 2>{}, std::integral_constant<int, 3>{});
    if (nfb <= 2 && nhb <= 4) return f(std::integral_constant<int, 2>{}, std::integral_constant<int, 4>{});
    if (nfb <= 4 && nhb <= 1) return f(std::integral_constant<int, 4>{}, std::integral_constant<int, 1>{});
    return cudaErrorNotSupported;
}

// Plan: geometry and slices (about one wave of resident CTAs over all channel
// tiles), for the workspace bound or the current device (plan_sms).
bool plan_wm(const TiledConv &p, dwconv_dtype dt, GeoWM &g, int &Zc, bool launch) {
    if ((dt != DWCONV_FP16 && dt != DWCONV_BF16) || p.FW < 8) return false;
    g = GeoWM{};
    g.tiles_h = (p.OHs + kWOTH - 1) / kWOTH;
    g.tiles_w = (p.OWs + kWOTW - 1) / kWOTW;
    g.ctiles = (p.C + kWCh - 1) / kWCh;
    const long long per = (long long)p.N * g.tiles_h * g.tiles_w;
    if (per >= (1LL << 30)) return false;
    g.per_ctile = (int)per;
    g.HR = kWOTH + p.FH - 1;
    bool ok = false;
    int resident = 1;  // CTAs per SM: two by the register bound, fewer if shared memory holds fewer
    with_shape(p.FH, p.FW, [&](auto nfb, auto nhb) {
        using C = CfgW<decltype(nfb)::value, decltype(nhb)::value>;
        g.x_bytes = (unsigned)g.HR * C::SWX * 16;
        ok = C::smem + 1024 <= 227 * 1024 && g.HR <= 256 && C::SWX <= 256;
        resident = std::max(1, std::min(2, (int)(plan_smem_per_sm(launch) / (C::smem + 2048))));
        return cudaSuccess;
    });
    if (!ok) return false;
    long long z = (long long)plan_sms(launch) * resident / g.ctiles;
    if (z > g.per_ctile) z = g.per_ctile;
    if (z < 1) z = 1;
    Zc = (int)z;
    return true;
}

template <typename T, int NFB, int NHB>
cudaError_t run_wm(const TiledConv &p, dwconv_dtype dt, const GeoWM &g, int Zc, float *part, cudaStream_t st) {
    using C = CfgW<NFB, NHB>;
    const size_t es = sizeof(T);
    const char *base = static_cast<const char *>(p.in) + ((size_t)p.in_off_h * p.Wf + p.in_off_w) * p.C * es;
    const uint64_t dims[4] = {(uint64_t)p.C, (uint64_t)p.Ws, (uint64_t)p.Hs, (uint64_t)p.N};
    uint64_t str[3];
    in_strides(p, es, str);
    const uint32_t box[4] = {(uint32_t)kWCh, (uint32_t)C::SWX, (uint32_t)g.HR, 1};
    const uint64_t ddims[4] = {(uint64_t)p.C, (uint64_t)p.OWs, (uint64_t)p.OHs, (uint64_t)p.N};
    const uint64_t mem_row = (uint64_t)(p.transpose ? p.OHs : p.OWs) * p.C * es, mem_col = (uint64_t)p.C * es;
    const uint64_t dstr[3] = {p.transpose ? mem_row : mem_col, p.transpose ? mem_col : mem_row,
                              (uint64_t)p.OHs * p.OWs * p.C * es};
    const uint32_t dbox[4] = {(uint32_t)kWCh, (uint32_t)kWOTW, (uint32_t)kWOTH, 1};
    CUtensorMap halo_map, dy_map;
    if (!encode_tmap_4d(&halo_map, dt, base, dims, str, box) || !encode_tmap_4d(&dy_map, dt, p.dy, ddims, dstr, dbox))
        return cudaErrorNotSupported;
    auto kern = tiled_mma_wgrad_kernel<T, NFB, NHB>;
    const int smem = (int)C::smem + 1024;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kWThreads, smem, nullptr);
    if (e != cudaSuccess) return e;
    kern<<<g.ctiles * Zc, kWThreads, smem, st>>>(halo_map, dy_map, p, g, part, Zc, device_error_word());
    note_launches(1);
    note_kernel("tiled_mma_wgrad");
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_wgrad_reduce(part, Zc, (long long)p.FH * p.FW * p.C, static_cast<float *>(p.out), st);
}

}  // namespace

#ifndef DWCONV_MMA_WGRAD
#define DWCONV_MMA_WGRAD 1  // 0: leave large-filter wgrad to the CUDA-core kernel
#endif

int tiled_mma_wgrad_slices(const TiledConv &p, dwconv_dtype dt) {
    GeoWM g;
    int Zc = 0;
    return DWCONV_MMA_WGRAD && plan_wm(p, dt, g, Zc, false) ? Zc : 0;
}

cudaError_t launch_tiled_mma_wgrad(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st) {
    GeoWM g;
    int Zc = 0;
    if (!DWCONV_MMA_WGRAD || !plan_wm(p, dt, g, Zc, true)) return cudaErrorNotSupported;
    return with_shape(p.FH, p.FW, [&](auto nfb, auto nhb) {
        constexpr int NFB = decltype(nfb)::value, NHB = decltype(nhb)::value;
        return dt == DWCONV_FP16 ? run_wm<__half, NFB, NHB>(p, dt, g, Zc, part, st)
                                 : run_wm<__nv_bfloat16, NFB, NHB>(p, dt, g, Zc, part, st);
    });
}

}  // namespace dwc
