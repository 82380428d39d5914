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
// Work: 8 channels (one per warp) x OTH-row, OTW-column bands of dy, 256
// threads.  A band of OTH dy rows reads OTH + FH - 1 x rows, so consecutive
// bands of an image column share all but OTH of them: each CTA walks an equal
// share of its channel tile's bands in order (column by column) and keeps the
// x rows in a ring in shared memory (channel-major, NPR >= NP pieces of OTH rows), so
// each step stages and transposes only the OTH new x rows (and the band's dy
// tile) instead of the whole halo.  Each image column a CTA enters starts with
// NP - 1 steps that fill the ring.  Per step one thread stages the new x rows
// and the dy tile by TMA into a ring of staging buffers (bounded waits);
// ldmatrix.trans + stmatrix build the channel-major copies -- dy twice, the
// second shifted by one column, so that every A pair is one aligned 32-bit
// load; each warp then runs its channel's MMAs with the NFB x NHB accumulator
// blocks in registers for the whole CTA, reading B from the ring at the band's
// offset (modulo the ring size).  Grid = channel tiles x accumulation slices;
// each CTA writes its slice of the partial sums and wgrad_reduce (direct.cu)
// sums the slices in a fixed order.
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
// dy rows, columns per band (measured on GB300: 4 x 64 beats 8 x 32 by 8-15 %,
// the wider tile wasting fewer Toeplitz products at its edges)
constexpr int kWOTH = DWCONV_WG_OTH, kWOTW = DWCONV_WG_OTW;
constexpr int kWStages = 3;  // staging buffers (new x rows + dy tile of one step each)

// Channel stride of a channel-major copy: 8 mod 16 halves, so that the 16-byte
// rows stmatrix writes for 8 channels fall in distinct bank quads.
constexpr int chan_stride(int v) { return v + ((8 - v % 16) + 16) % 16; }

template <int NFB, int NHB>
struct CfgW {
    static constexpr int FWMAX = 16 * NFB, FHMAX = 8 * NHB;
    // x columns OTW + FW - 1 rounded up to whole 16-column groups, NG of them at most.
    static constexpr int NG = (kWOTW + FWMAX - 1 + 15) / 16;
    static constexpr int SWX = 16 * NG;
    // Diagonals d = grp - fb whose blocks meet a dy column of the tile: 0 <= d < ND.
    static constexpr int ND = NG < (kWOTW + 14) / 16 + 1 ? NG : (kWOTW + 14) / 16 + 1;
    // x rows one band's MMAs read, from the band's first x row (the last
    // block's surplus rows only reach unused accumulator columns).
    static constexpr int TXR = kWOTH + FHMAX - 1;
    static constexpr int NP = (TXR + kWOTH - 1) / kWOTH;  // pieces of OTH x rows a window spans
    // T_x row stride: 8 rows of a B load fall in distinct bank quads.
    static constexpr int RSX = SWX % 16 == 8 ? SWX : SWX + ((8 - SWX % 16 + 16) % 16);
    // T_dy: dy column e sits at LM + e (copy 1: e + 1); the A loads reach e
    // from -15 to 16 ND - 1, the transposes write up to OTW + 7; 8 mod 16
    // halves per row keeps the two copies' A loads in disjoint banks.
    static constexpr int LM = 16;
    static constexpr int DW = chan_stride(LM + (16 * ND > kWOTW + 8 ? 16 * ND : kWOTW + 8) + 1);
    static constexpr int CSD = chan_stride(2 * kWOTH * DW);  // two copies per channel
    static constexpr unsigned x_bytes = (unsigned)kWOTH * SWX * 16;  // one piece: OTH rows x SWX cols x 8 ch
    static constexpr unsigned dy_bytes = kWOTH * kWOTW * 16;
    static constexpr unsigned dy_off = align1k(x_bytes);  // dy box within a stage
    static constexpr unsigned stage = dy_off + align1k(dy_bytes);
    static constexpr unsigned tx_off = kWStages * stage;
    static constexpr unsigned td_bytes = kWCh * CSD * 2;
    static constexpr unsigned smem_with(int pieces) {
        return tx_off + kWCh * chan_stride(pieces * kWOTH * RSX) * 2 + td_bytes + 16;
    }
    // Ring pieces: rounded up to a multiple of 8 rows when two CTAs still fit
    // an SM, so that the 8 rows of a B load that wraps around the ring's end
    // stay in distinct bank quads too.
    static constexpr int NP8 = ((NP * kWOTH + 7) / 8 * 8) / kWOTH;
    static constexpr int NPR = 2 * (smem_with(NP8) + 2048) <= 228 * 1024 ? NP8 : NP;
    static constexpr int R = NPR * kWOTH;  // ring rows
    static constexpr int CSX = chan_stride(R * RSX);
    static constexpr unsigned td_off = tx_off + kWCh * CSX * 2;  // 16-byte aligned, as stmatrix needs
    static constexpr unsigned zero_off = td_off + td_bytes;
    static constexpr unsigned smem = zero_off + 16;
    // Small accumulator shapes leave room for three CTAs per SM.
    static constexpr int kMinBlocks = NFB * NHB <= 2 ? 3 : 2;
};

// Bands of a channel tile, numbered column by column: band f is band
// f mod tiles_h of image column f / tiles_h (column = image n x column tile).
struct GeoWM {
    int tiles_h, tiles_w, ctiles;
    int total;  // N * tiles_w * tiles_h
};

// A CTA's walk over its band range [f0, f1): one segment per image column
// it meets, each NP - 1 ring-filling steps (x only) and then one step per
// band.  Step k of a segment stages x piece k (rows r0 + k OTH .., with
// r0 = b0 OTH - pad); steps k >= NP - 1 also stage the dy tile of band
// b0 + k - (NP - 1) and run its MMAs on the ring window of pieces
// k - (NP - 1) .. k.
struct Cursor {
    int f;       // first band of the segment (flat); f >= f1 when done
    int n, twi;  // image, column tile
    int b0, b1;  // band range of the segment within the column
    int k;       // step within the segment
};

__device__ __forceinline__ void seg_start(Cursor &c, const GeoWM &g, int f, int f1) {
    c.f = f;
    c.k = 0;
    if (f >= f1) return;
    const int col = f / g.tiles_h;
    c.n = col / g.tiles_w;
    c.twi = col % g.tiles_w;
    c.b0 = f - col * g.tiles_h;
    c.b1 = min(g.tiles_h, f1 - col * g.tiles_h);
}

template <typename T, int NFB, int NHB>
__global__ void __launch_bounds__(kWThreads, CfgW<NFB, NHB>::kMinBlocks)
    tiled_mma_wgrad_kernel(const __grid_constant__ CUtensorMap halo_map, const __grid_constant__ CUtensorMap dy_map,
                           TiledConv p, GeoWM g, float *__restrict__ part, int Zc, unsigned *err) {
    using C = CfgW<NFB, NHB>;
    constexpr int NG = C::NG, NP = C::NP, NS = kWStages;
    // 128-byte alignment (the staging buffers sit at 1 KB multiples from it)
    // is what the unswizzled TMA boxes need.
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[NS];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int gq = lane / 4, t4 = lane % 4;
    const int tr = lane % 8, tj = lane / 8;
    const unsigned s_addr = smem_addr(smem_raw);
    const unsigned tx_addr = s_addr + C::tx_off, td_addr = s_addr + C::td_off, zero_addr = s_addr + C::zero_off;
    const int ctile = blockIdx.x / Zc, z = blockIdx.x % Zc;

    // Zero T_x and T_dy once: T_dy's margins are never written again.
    for (unsigned i = tid; i < (C::zero_off + 16 - C::tx_off) / 16; i += kWThreads)
        reinterpret_cast<uint4 *>(smem_raw + C::tx_off)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int b = 0; b < NS; ++b) mbar_init(&bars[b], 1);
        mbar_fence_init();
    }
    __syncthreads();

    // This CTA's bands: an equal share of the channel tile's, in order.
    const int f0 = (int)((long long)g.total * z / Zc), f1 = (int)((long long)g.total * (z + 1) / Zc);
    auto next = [&](Cursor &c) {
        if (++c.k == NP - 1 + (c.b1 - c.b0)) seg_start(c, g, c.f + (c.b1 - c.b0), f1);
    };
    auto issue = [&](const Cursor &c, int b) {
        const bool band = c.k >= NP - 1;
        unsigned char *dst = smem_raw + b * C::stage;
        mbar_arrive_expect_tx(&bars[b], C::x_bytes + (band ? C::dy_bytes : 0u));
        tma_load_4d(dst, &halo_map, ctile * kWCh, c.twi * kWOTW - p.pad_w, (c.b0 + c.k) * kWOTH - p.pad_h, c.n,
                    &bars[b]);
        if (band)
            tma_load_4d(dst + C::dy_off, &dy_map, ctile * kWCh, c.twi * kWOTW, (c.b0 + c.k - (NP - 1)) * kWOTH,
                        c.n, &bars[b]);
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
    const int q2 = gq & 1;
    const unsigned a_lane = td_c + 2u * (unsigned)(q2 * kWOTH * C::DW + C::LM + 2 * t4 - gq + q2);
    // B pair: x row (band row i + 8 hb + gq of the window), columns 8 grp + 2t4, +1.
    const unsigned b_col = tx_c + 2u * (unsigned)(2 * t4);

    Cursor ld, cur;
    seg_start(ld, g, f0, f1);
    seg_start(cur, g, f0, f1);
    int issued = 0;  // steps thread 0 has issued
    if (tid == 0)
        for (; issued < NS - 1 && ld.f < f1; ++issued, next(ld)) issue(ld, issued);
    for (int s = 0; cur.f < f1; ++s, next(cur)) {
        if (tid == 0 && ld.f < f1) {
            issue(ld, (s + NS - 1) % NS);  // the buffer of step s - 1, free since its first barrier
            next(ld);
            ++issued;
        }
        if (!mbar_wait(&bars[s % NS], (s / NS) & 1)) {
            // Give up: thread 0 lets the copies it issued land (bounded) before leaving.
            report_timeout(err);
            if (tid == 0)
                for (int j = s + 1; j < issued; ++j) mbar_wait(&bars[j % NS], (j / NS) & 1);
            return;
        }
        const unsigned sx = s_addr + (s % NS) * C::stage;
        const unsigned sd = sx + C::dy_off;
        const bool band = cur.k >= NP - 1;
        // New x rows [OTH][SWX][8 ch] -> ring slot k mod NPR of T_x[ch][row][col],
        // four 8-pixel blocks per step (lane (tr, tj) addresses pixel tr of block tj).
        {
            constexpr int CB = C::SWX / 8;  // 8-pixel blocks per row
            constexpr int nb = kWOTH * CB;
            const int slot = (cur.k % C::NPR) * kWOTH;
            for (int m0 = warp * 4; m0 < nb; m0 += kWThreads / 8) {
                const int m = min(m0 + tj, nb - 1);
                const int row = m / CB, col0 = (m % CB) * 8;
                unsigned v0, v1, v2, v3;
                ldsm_x4_trans(v0, v1, v2, v3, sx + (unsigned)((row * C::SWX + col0 + tr) * 16));
                stsm_x4(tx_addr + 2u * (unsigned)(tr * C::CSX + (slot + row) * C::RSX + col0), v0, v1, v2, v3);
            }
        }
        // dy: copy 0 at columns LM + j, copy 1 (dy[j - 1]) at LM + j; copy 1's
        // blocks start one pixel early, with the zero pixel outside the tile.
        if (band) {
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
        __syncthreads();  // the new ring rows and T_dy are ready; this staging buffer is free
        if (!band) continue;

        // MMAs of this warp's channel, 16 x columns each (m16n8k16).  A of
        // block fb, group grp depends on the diagonal d = grp - fb only: dy
        // columns e0 = 16 d + 2t4 - gq (a0), e0 - 8 (a1, M rows 8-15), e0 + 8
        // (a2, k 8-15) and e0 again (a3: rows 8-15 and k 8-15 cancel), and
        // a1 of diagonal d is a2 of diagonal d - 1; so a row loads 2 ND + 1
        // pairs.  Blocks with d outside [0, ND) meet no dy column of the tile
        // and are skipped at compile time.  B of block hb comes from the
        // window's x row i + 8 hb + gq, ring row (window start + that) mod R.
        const int base = ((cur.k - (NP - 1)) % C::NPR) * kWOTH;
#pragma unroll 1
        for (int i = 0; i < kWOTH; ++i) {
            constexpr int ND = C::ND;
            const unsigned arow = a_lane + 2u * (unsigned)(i * C::DW);
            unsigned a0[ND], a2[ND], a1first;
            asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(a1first) : "r"(arow - 16u));  // 8 columns left
#pragma unroll
            for (int d = 0; d < ND; ++d) {
                asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(a0[d]) : "r"(arow + 32u * d));
                asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(a2[d]) : "r"(arow + 32u * d + 16u));  // 8 right
            }
            unsigned brow[NHB];
#pragma unroll
            for (int hb = 0; hb < NHB; ++hb) {
                int rr = base + i + 8 * hb + gq;
                if (rr >= C::R) rr -= C::R;
                brow[hb] = b_col + 2u * (unsigned)(rr * C::RSX);
            }
#pragma unroll
            for (int grp = 0; grp < NG; ++grp) {
                if (grp - (NFB - 1) >= ND) continue;  // every block of this group skipped
                unsigned b[NHB][2];
#pragma unroll
                for (int hb = 0; hb < NHB; ++hb) {
                    const unsigned ba = brow[hb] + 32u * (unsigned)grp;
                    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(b[hb][0]) : "r"(ba));
                    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(b[hb][1]) : "r"(ba + 16u));
                }
#pragma unroll
                for (int fb = 0; fb < NFB; ++fb) {
                    const int d = grp - fb;
                    if (d < 0 || d >= ND) continue;
                    const unsigned a1 = d == 0 ? a1first : a2[d > 0 ? d - 1 : 0];
#pragma unroll
                    for (int hb = 0; hb < NHB; ++hb)
                        MmaOp<T>::run(acc[fb][hb], a0[d], a1, a2[d], a0[d], b[hb][0], b[hb][1]);
                }
            }
        }
        __syncthreads();  // every warp is done with this window and T_dy
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

// Plan for the workspace bound or the current device (plan_sms): at most one
// wave of resident CTAs over all channel tiles, each with an equal range of
// bands.  A range pays NP - 1 ring-filling steps (x only, taken as a quarter
// of a band step) per image column it meets; the slice count with the
// shortest worst range wins, the most slices on ties.
bool plan_wm(const TiledConv &p, dwconv_dtype dt, GeoWM &g, int &Zc, bool launch) {
    if ((dt != DWCONV_FP16 && dt != DWCONV_BF16) || p.FW < 8) return false;
    g = GeoWM{};
    g.tiles_h = (p.OHs + kWOTH - 1) / kWOTH;
    g.tiles_w = (p.OWs + kWOTW - 1) / kWOTW;
    g.ctiles = (p.C + kWCh - 1) / kWCh;
    const long long total = (long long)p.N * g.tiles_w * g.tiles_h;
    if (total >= (1LL << 30)) return false;
    g.total = (int)total;
    bool ok = false;
    int resident = 1, fill = 0;  // CTAs per SM; ring-filling steps per segment
    const cudaError_t e = with_shape(p.FH, p.FW, [&](auto nfb, auto nhb) {
        constexpr int NFB = decltype(nfb)::value, NHB = decltype(nhb)::value;
        using C = CfgW<NFB, NHB>;
        ok = C::smem <= 227 * 1024 && C::SWX <= 256;
        fill = C::NP - 1;
        // The bound: what shared memory and the register bound allow; at a
        // launch: the occupancy the device reports for this kernel.
        resident = std::max(1, std::min(C::kMinBlocks, (int)(plan_smem_per_sm(launch) / (C::smem + 2048))));
        if (!ok || !launch) return cudaSuccess;
        const void *kern = dt == DWCONV_FP16 ? reinterpret_cast<const void *>(tiled_mma_wgrad_kernel<__half, NFB, NHB>)
                                             : reinterpret_cast<const void *>(tiled_mma_wgrad_kernel<__nv_bfloat16, NFB, NHB>);
        int per_sm = 0;
        const cudaError_t k = kernel_setup(kern, kWThreads, C::smem, &per_sm);
        if (k == cudaSuccess) resident = std::max(1, std::min(resident, per_sm));
        return k;
    });
    if (e != cudaSuccess || !ok) return false;
    const long long target = std::min(total, std::max(1LL, (long long)plan_sms(launch) * resident / g.ctiles));
    long long best = -1;
    for (long long z = target; z >= 1; --z) {
        const long long L = (total + z - 1) / z;           // bands of the longest range
        const long long segs = (L + g.tiles_h - 2) / g.tiles_h + 1;  // columns it can meet
        const long long cost = 4 * L + fill * segs;
        if (best < 0 || cost < best) {
            best = cost;
            Zc = (int)z;
        }
        if (4 * L > best) break;  // fewer slices only lengthen the ranges
    }
    if (launch) {
        // The partial-sum workspace was sized by the bound plan: never more slices.
        GeoWM gb;
        int zb = 0;
        if (!plan_wm(p, dt, gb, zb, false)) return false;
        Zc = std::min(Zc, zb);
    }
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
    const uint32_t box[4] = {(uint32_t)kWCh, (uint32_t)C::SWX, (uint32_t)kWOTH, 1};  // one ring piece
    const uint64_t ddims[4] = {(uint64_t)p.C, (uint64_t)p.OWs, (uint64_t)p.OHs, (uint64_t)p.N};
    const uint64_t mem_row = (uint64_t)(p.transpose ? p.OHs : p.OWs) * p.C * es, mem_col = (uint64_t)p.C * es;
    const uint64_t dstr[3] = {p.transpose ? mem_row : mem_col, p.transpose ? mem_col : mem_row,
                              (uint64_t)p.OHs * p.OWs * p.C * es};
    const uint32_t dbox[4] = {(uint32_t)kWCh, (uint32_t)kWOTW, (uint32_t)kWOTH, 1};
    CUtensorMap halo_map, dy_map;
    if (!encode_tmap_4d(&halo_map, dt, base, dims, str, box) || !encode_tmap_4d(&dy_map, dt, p.dy, ddims, dstr, dbox))
        return cudaErrorNotSupported;
    auto kern = tiled_mma_wgrad_kernel<T, NFB, NHB>;
    const int smem = (int)C::smem;
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
