// Tensor-core forward pass and stride-1 input gradient for 16-bit data and
// large filters, maps at least 17 columns wide.  Compiled filter heights: every
// odd height from 9 to 31 with the number of 16-input blocks its square filter
// needs (tiled_mma_large.cu and tiled_mma_large_h*.cu; a filter of another
// width runs here when it needs the same number of blocks), and 5 rows with 42
// to 57 columns (the strips of factorised large kernels, also taken transposed
// for 42-57 x 5).
//
// The packing is the one of the small-filter kernel (Flash-DWC §4.2): for a
// filter row fh, 8 consecutive outputs of one output row read a window of
// 8 + FW - 1 inputs, so the Toeplitz band B[k][n] = w[fh][k - n] is split into
// NKB = ceil((FW + 7) / 16) blocks of 16 inputs, and one m16n8k16 MMA per
// block takes 16 such groups of 8 outputs:
//
//   Y[group m][n] += sum_kb sum_{k<16} X[ih][8 j_m + 16 kb + k] * w[fh][16 kb + k - n].
//
// For a 31-wide filter 248 of the 384 products of the three blocks are taps
// of the filter (65 %, against 44 % for 7x7).
//
// Work unit: 8 channels (one per warp) x OTH = 2 * 7 * (8/G) output rows x
// OTW = 8G columns of one image, 256 threads.
//   1. one TMA copy stages the NHWC halo (16-byte pixels, zeros outside the
//      input); the next unit's copy is issued as soon as this one has been
//      transposed;
//   2. ldmatrix.trans + stmatrix transpose it into T[channel][row][column];
//   3. per filter block kb the warp keeps the B fragments of all FH filter
//      rows in registers and walks the input rows x once: the A operand of
//      input row x (one ldmatrix.x4) serves the MMAs (row set j, filter row
//      x - j RB) of all 7 row sets, whose accumulators stay in registers over
//      all blocks and filter rows (fp32, bias added once at the start);
//   4. the results, rounded to 16 bits, go to an NHWC output tile that leaves
//      by TMA tensor store, clipped at the tensor edges.
#pragma once

#include "mma_common.cuh"

namespace dwc {
namespace {

using namespace tiled;
using namespace mma;

constexpr int kLCh = 8;         // channels per work unit, one per warp
constexpr int kLThreads = 256;  // 8 warps
constexpr int kLNB = 7;         // MMA row sets per work unit

template <int FH, int NKB, int G>
struct CfgL {
    static constexpr int RB = 8 / G;                        // output rows of one 8-row M block
    static constexpr int DH = kLNB * RB;                    // rows between the two M blocks
    static constexpr int OTH = 2 * DH, OTW = 8 * G;         // output tile
    static constexpr int HR = OTH + FH - 1;                 // staged halo rows
    static constexpr int SW = 8 * G - 8 + 16 * NKB;         // staged halo columns
    static constexpr int CB = SW / 8;                       // 8-column blocks of a row
    static constexpr int RS = SW, CS = channel_stride(HR * RS);
    static constexpr int FP = 16 * NKB + 8;                 // halves of one padded filter row copy
    static constexpr unsigned s_bytes = HR * SW * 16;       // one staged pixel = 8 channels
    static constexpr unsigned t_off = align1k(s_bytes);
    static constexpr unsigned o_off = t_off + align1k(kLCh * CS * 2);
    static constexpr unsigned f_off = o_off + align1k(OTH * OTW * 16);
    static constexpr unsigned smem = f_off + kLCh * FH * 2 * FP * 2;  // + 1 KB alignment slack
    static_assert(SW % 8 == 0, "16-byte T rows");
};

// FUSE: the fused forward pass (Flash-DWC §5.2) compiled in -- the BN+Act
// prologue during the transposition, the affine+activation epilogue on the
// fp32 sums; separate instances keep the plain passes' register allocation.
template <typename T, int FH, int NKB, int G, bool FUSE>
__global__ void __launch_bounds__(kLThreads, 1)
    tiled_mma_large_kernel(const __grid_constant__ CUtensorMap halo_map,
                           const __grid_constant__ CUtensorMap out_map, TiledConv p, GeoM g, unsigned *err) {
    using C = CfgL<FH, NKB, G>;
    constexpr int RB = C::RB, DH = C::DH;
    constexpr int NQ = (kLNB - 1) * RB + FH;  // A operands (input row positions) per block
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    __shared__ __align__(8) uint64_t bar;
    using Op = MmaOp<T>;

    unsigned char *smem_raw = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int gq = lane / 4, t4 = lane % 4;
    unsigned char *S = smem_raw;                 // [HR][SW][8]
    const unsigned s_addr = smem_addr(S);
    const unsigned t_addr = s_addr + C::t_off;   // [8][CS]
    const unsigned o_addr = s_addr + C::o_off;   // [OTH][OTW][8]
    T *F = reinterpret_cast<T *>(smem_raw + C::f_off);  // [8][FH][2][FP]
    const unsigned f_addr = s_addr + C::f_off;
    const T *wg = static_cast<const T *>(p.w);

    const int u_begin = (int)((long long)g.units * blockIdx.x / gridDim.x);
    const int u_end = (int)((long long)g.units * (blockIdx.x + 1) / gridDim.x);

    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();

    Unit ld = decode(g, u_begin), cur = ld;
    auto issue = [&]() {
        mbar_arrive_expect_tx(&bar, C::s_bytes);
        tma_load_4d(S, &halo_map, ld.ctile * kLCh, ld.twi * C::OTW - p.pad_w, ld.band * C::OTH - p.pad_h,
                    ld.group, &bar);
        advance(g, g.groups, ld);
    };
    if (tid == 0 && u_begin < u_end) issue();

    // A operand of input row x, block kb: one ldmatrix.x4; matrix j holds M
    // rows 8(j%2)..+7 (window i % G of input row x + i / G + DH (j%2)) and k
    // 8(j/2)..+7.
    const int mj = lane / 8, mi = lane % 8;
    const unsigned a_lane =
        t_addr + 2u * (warp * C::CS + ((mj & 1) * DH + mi / G) * C::RS + 8 * (mi % G) + 8 * (mj >> 1));
    // B pair of lane (gq, t4) in block kb: w[16 kb + 2t4 - gq (+1)], read from
    // the padded copy q = gq & 1 (copy q holds w[i + q - 8] at index i), where
    // it is 32-bit aligned.
    const int b_off = 2 * t4 - gq + 8 - (gq & 1);
    const unsigned b_lane = f_addr + 2u * ((warp * FH * 2 + (gq & 1)) * C::FP + b_off);
    // Transposition: lane (tr, tj) addresses row tr of matrix tj of a step.
    const int tr = lane % 8, tj = lane / 8;
    // Output: position (row gq / G (+ DH), column 8 (gq % G) + 2t4 + e); the
    // two columns go out in gq-parity order (4-way instead of 8-way conflicts).
    const unsigned o_lane = o_addr + 2u * (((gq / G) * C::OTW + 8 * (gq % G) + 2 * t4) * kLCh + warp);

    int loaded_ctile = -1;
    float bias_c = 0.f;
    for (int u = u_begin, k = 0; u < u_end; ++u, ++k, advance(g, g.groups, cur)) {
        if (cur.ctile != loaded_ctile) {
            // Every warp finished reading F (previous unit) before the last
            // barrier.  Zero the table, then scatter the filter: value (fh, fw)
            // of channel c goes to index fw + 8 - q of copy q of row fh (rows
            // rotated by 180 degrees for the input gradient).
            loaded_ctile = cur.ctile;
            constexpr int kWords = kLCh * FH * 2 * C::FP / 8;  // 16-byte words
            for (int i = tid; i < kWords; i += kLThreads) reinterpret_cast<uint4 *>(F)[i] = make_uint4(0, 0, 0, 0);
            __syncthreads();
            // Loads per thread in flight at a time: one at a time, the rebuild
            // took 7 % of a 31x31 forward pass.  Measured on GB300: 8 for most
            // heights; 32 (the whole table in one batch) from 29 rows on (31x31
            // 2-3 % faster, 29x29 equal; slower for smaller filters).
            const int nw = kLCh * FH * p.FW;
            constexpr int kBatch = FH >= 29 ? 32 : 8;
            for (int i0 = tid; i0 < nw; i0 += kBatch * kLThreads) {
                T v[kBatch];
                int at[kBatch];  // index of copy 0 in F, or -1
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int i = i0 + b * kLThreads;
                    at[b] = -1;
                    if (i >= nw) continue;
                    const int c = i % kLCh, t = i / kLCh, fw = t % p.FW, fh = t / p.FW;
                    const int cc = cur.ctile * kLCh + c;
                    if (cc >= p.C) continue;
                    // Transposed view: kernel tap (fh, fw) is memory tap (fw, fh).
                    const int mt = p.transpose ? fw * FH + fh : t;
                    v[b] = __ldg(wg + (size_t)mt * p.C + cc);
                    const int dfh = p.flip ? FH - 1 - fh : fh, dfw = p.flip ? p.FW - 1 - fw : fw;
                    at[b] = (c * FH + dfh) * 2 * C::FP + dfw + 8;
                }
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (at[b] >= 0) {
                        F[at[b]] = v[b];             // copy 0
                        F[at[b] + C::FP - 1] = v[b]; // copy 1
                    }
            }
            const int cc = cur.ctile * kLCh + warp;
            bias_c = (p.bias && cc < p.C) ? p.bias[cc] : 0.f;
        }
        if (!mbar_wait(&bar, k & 1)) {
            // Thread 0 lets the copies in flight end (bounded) before leaving.
            report_timeout(err);
            if (tid == 0) {
                mbar_wait(&bar, k & 1);
                asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
            }
            return;
        }
        // Transpose S[row][col][8 ch] -> T[ch][row][col], four 8-column blocks
        // per step; the last step repeats its final block where the count is
        // not a multiple of 4 (same data to the same place).
        // With the BN+Act prologue, lane (gq, t4) holds channel gq of
        // columns 2t4, 2t4+1 of block m0 + j in register j; positions outside
        // the input are padding of x' and stay zero.
        auto transpose = [&](auto pre) {
            constexpr int PA = decltype(pre)::value;  // activation, or -1: no prologue
            float2 s2 = make_float2(1.f, 1.f), t2 = make_float2(0.f, 0.f);
            unsigned cmask = 0;  // bit 2i + e: column 8i + 2t4 + e lies inside the input
            if constexpr (PA >= 0) {
                const int c = cur.ctile * kLCh + gq;
                if (c < p.C) {
                    const Affine a = affine_in(p.fz, c);
                    s2 = make_float2(a.s, a.s);
                    t2 = make_float2(a.t, a.t);
                }
                static_assert(C::CB <= 16, "column mask of 32 bits");
                const int iw0 = cur.twi * C::OTW - p.pad_w + 2 * t4;
#pragma unroll
                for (int i = 0; i < C::CB; ++i)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int iw = iw0 + 8 * i + e;
                        cmask |= (iw >= 0 && iw < p.Ws ? 1u : 0u) << (2 * i + e);
                    }
            }
            constexpr int kBlocks = C::HR * C::CB, kStride = kLThreads / 8;
            auto src = [&](int m0) {
                const int m = min(m0 + tj, kBlocks - 1);
                return s_addr + (unsigned)(((m / C::CB) * C::SW + (m % C::CB) * 8 + tr) * 16);
            };
            auto dst = [&](int m0) {
                const int m = min(m0 + tj, kBlocks - 1);
                return t_addr + 2u * (tr * C::CS + (m / C::CB) * C::RS + (m % C::CB) * 8);
            };
            if constexpr (PA < 0) {
                // Two steps per iteration: both loads are in flight before the stores.
                int m0 = warp * 4;
                for (; m0 + kStride < kBlocks; m0 += 2 * kStride) {
                    unsigned v[2][4];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        ldsm_x4_trans(v[u][0], v[u][1], v[u][2], v[u][3], src(m0 + u * kStride));
#pragma unroll
                    for (int u = 0; u < 2; ++u) stsm_x4(dst(m0 + u * kStride), v[u][0], v[u][1], v[u][2], v[u][3]);
                }
                for (; m0 < kBlocks; m0 += kStride) {
                    unsigned v[4];
                    ldsm_x4_trans(v[0], v[1], v[2], v[3], src(m0));
                    stsm_x4(dst(m0), v[0], v[1], v[2], v[3]);
                }
            } else {
                for (int m0 = warp * 4; m0 < kBlocks; m0 += kStride) {
                    unsigned v[4];
                    ldsm_x4_trans(v[0], v[1], v[2], v[3], src(m0));
                    // Blocks m0..m0+3 (clamped to the last): row r, column chunk ch.
                    int r = m0 / C::CB, ch = m0 - r * C::CB;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (j > 0 && m0 + j < kBlocks && ++ch == C::CB) ch = 0, ++r;
                        const int ih = cur.band * C::OTH - p.pad_h + r;
                        const unsigned m2 = ih >= 0 && ih < p.Hs ? (cmask >> (2 * ch)) & 3u : 0u;
                        const unsigned keep = (m2 & 1u ? 0x0000FFFFu : 0u) | (m2 & 2u ? 0xFFFF0000u : 0u);
                        v[j] = prologue_packed<T, PA>(v[j], s2, t2) & keep;
                    }
                    stsm_x4(dst(m0), v[0], v[1], v[2], v[3]);
                }
            }
        };
        if (FUSE && p.fz.pre())
            with_act(p.fz.in_act, transpose);
        else
            transpose(std::integral_constant<int, -1>{});
        if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
        __syncthreads();  // T and F ready, S and the output tile free
        if (tid == 0 && u + 1 < u_end) issue();

        float d[kLNB][4];
#pragma unroll
        for (int j = 0; j < kLNB; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = bias_c;
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb) {
            unsigned bf[FH][2];
#pragma unroll
            for (int fh = 0; fh < FH; ++fh) {
                const unsigned a = b_lane + 2u * (fh * 2 * C::FP + 16 * kb);
                asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(bf[fh][0]) : "r"(a));
                asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(bf[fh][1]) : "r"(a + 16));
            }
            unsigned A[2][4];
            ldsm_x4(A[0][0], A[0][1], A[0][2], A[0][3], a_lane + 2u * (16 * kb));
#pragma unroll
            for (int x = 0; x < NQ; ++x) {
                if (x + 1 < NQ)
                    ldsm_x4(A[(x + 1) & 1][0], A[(x + 1) & 1][1], A[(x + 1) & 1][2], A[(x + 1) & 1][3],
                            a_lane + 2u * ((x + 1) * C::RS + 16 * kb));
#pragma unroll
                for (int j = 0; j < kLNB; ++j) {
                    const int fh = x - j * RB;
                    if (fh >= 0 && fh < FH)
                        Op::run(d[j], A[x & 1][0], A[x & 1][1], A[x & 1][2], A[x & 1][3], bf[fh][0], bf[fh][1]);
                }
            }
        }

        if (FUSE && p.fz.post()) {
            const int cc = cur.ctile * kLCh + warp;
            const Affine a = cc < p.C ? affine_out(p.fz, cc) : Affine{1.f, 0.f};
            with_act(p.fz.out_act, [&](auto act) {
#pragma unroll
                for (int j = 0; j < kLNB; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) d[j][e] = activate(fmaf(a.s, d[j][e], a.t), decltype(act)::value);
            });
        }

        // Output tile [OTH][OTW][8 ch]: this lane's channel, 2 bytes per position.
        const bool odd = gq & 1;
#pragma unroll
        for (int j = 0; j < kLNB; ++j)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const unsigned row = 2u * ((j * RB + half * DH) * C::OTW * kLCh);
                const unsigned short v0 = Op::bits(d[j][2 * half]), v1 = Op::bits(d[j][2 * half + 1]);
                asm volatile("st.shared.b16 [%0], %1;\n" ::"r"(o_lane + row + (odd ? 2 * kLCh : 0)),
                             "h"(odd ? v1 : v0)
                             : "memory");
                asm volatile("st.shared.b16 [%0], %1;\n" ::"r"(o_lane + row + (odd ? 0 : 2 * kLCh)),
                             "h"(odd ? v0 : v1)
                             : "memory");
            }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncthreads();  // output tile complete; every warp is done with T and F
        if (tid == 0) {
            asm volatile(
                "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];\n" ::"l"(
                    reinterpret_cast<uint64_t>(&out_map)),
                "r"(cur.ctile * kLCh), "r"(cur.twi * C::OTW), "r"(cur.band * C::OTH), "r"(cur.group), "r"(o_addr)
                : "memory");
            asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
        }
    }
    if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}

template <typename T, int FH, int NKB, int G, bool FUSE>
cudaError_t run_large(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    using C = CfgL<FH, NKB, G>;
    if (C::smem + 1024 > 227 * 1024) return cudaErrorNotSupported;
    GeoM g{};
    g.tiles_h = (p.OHs + C::OTH - 1) / C::OTH;
    g.tiles_w = (p.OWs + C::OTW - 1) / C::OTW;
    g.groups = p.N;
    const long long per = (long long)p.N * g.tiles_w * g.tiles_h;
    const long long units = per * ((p.C + kLCh - 1) / kLCh);
    if (units >= (1LL << 30)) return cudaErrorNotSupported;
    g.per_ctile = (int)per;
    g.units = (int)units;
    const size_t es = sizeof(T);
    const char *base = static_cast<const char *>(p.in) + ((size_t)p.in_off_h * p.Wf + p.in_off_w) * p.C * es;
    const uint64_t dims[4] = {(uint64_t)p.C, (uint64_t)p.Ws, (uint64_t)p.Hs, (uint64_t)p.N};
    uint64_t str[3];
    in_strides(p, es, str);
    const uint32_t box[4] = {(uint32_t)kLCh, (uint32_t)C::SW, (uint32_t)C::HR, 1};
    const uint32_t obox[4] = {(uint32_t)kLCh, (uint32_t)C::OTW, (uint32_t)C::OTH, 1};
    CUtensorMap map, omap;
    if (!encode_tmap_4d(&map, dt, base, dims, str, box) || !make_out_map(&omap, p, dt, es, obox, 0))
        return cudaErrorNotSupported;
    auto kern = tiled_mma_large_kernel<T, FH, NKB, G, FUSE>;
    int per_sm = 0;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kLThreads, C::smem + 1024, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const int grid = (int)std::min<long long>(g.units, (long long)sm_count() * per_sm);
    kern<<<grid, kLThreads, C::smem + 1024, st>>>(map, omap, p, g, device_error_word());
    note_launches(1);
    note_kernel("tiled_mma_large");
    return cudaGetLastError();
}

template <typename T, int FH, int NKB, bool FUSE>
cudaError_t large_by_width(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (p.OWs > 32) return run_large<T, FH, NKB, 8, FUSE>(p, dt, st);
    if (p.OWs > 16) return run_large<T, FH, NKB, 4, FUSE>(p, dt, st);
    return cudaErrorNotSupported;
}

}  // namespace

// Plain (unfused) instances of further filter heights, one translation unit
// each so that they compile in parallel; each returns cudaErrorNotSupported
// for a shape it does not cover.
cudaError_t launch_mma_large_h1(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);
cudaError_t launch_mma_large_h2(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);
cudaError_t launch_mma_large_h3(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);

}  // namespace dwc
