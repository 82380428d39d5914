// Tensor-core forward pass and stride-1 input gradient for 16-bit data and
// 3x3, 5x5 and 7x7 filters.
//
// The GEMV of one channel (Flash-DWC §2.1) is packed into dense MMAs as in
// Flash-DWC §4.2: 8 consecutive outputs of one output row ("a group") read a
// window of 16 consecutive inputs, and for one filter row fh
//
//   Y[group m][n] += sum_{k<16} A[m][k] * B[k][n],   A[m][k] = X[ih][8j_m + k],
//                                                    B[k][n] = w[fh][k - n] (0 outside [0, FW)),
//
// a 16 x 8 Toeplitz band of the filter row.  One warp-level mma.sync
// m16n8k16 (bf16/fp16 in, fp32 accumulate) takes 16 groups at once, in two
// blocks of 8 M rows; a block is G groups of each of 8/G output rows spaced G
// apart (G = 8 on maps wider than 32 columns, 4 above 16, 2 above 8): with
// that spacing the 8 row addresses of every operand matrix fall in distinct
// shared-memory banks (adjacent rows put two of them in one bank for G < 8).
// A channel's output block needs FH such MMAs (one per filter row); the
// accumulator stays in registers across them, so every partial sum is kept in
// fp32 and the bias is added once, at the start.
//
// Work unit: 32 channels x OTW = 8G columns of NI images, 256 threads, each
// warp 4 channels; contiguous unit ranges per CTA.  With NI = 1 (maps more
// than 16 columns wide) the unit is OTH = 2 * KNB * 8/G rows of one image and
// M rows 8-15 cover the rows half a tile below rows 0-7; with NI = 2 (narrow
// maps, few rows) it is OTH = KNB * 8/G rows of two images and M rows 8-15
// cover the same rows of the second image.
//   1. one TMA copy stages the NHWC input halo in shared memory with the
//      64-byte swizzle (zeros outside the input: padding is generated); with
//      room for two staging buffers the next two units' loads are in flight;
//   2. ldmatrix.trans + stmatrix transpose it into a channel-major buffer
//      T[channel][row][column], in which the 8 windows of an 8-row matrix of
//      an MMA operand are 8 rows of 16 bytes (one ldmatrix matrix);
//   3. the A operands of the KNB row sets x FH filter rows overlap: MMA (row
//      set j, filter row fh) reads rows from x = base(j) + fh on, so the
//      operand of x (one ldmatrix.x4) serves every (j, fh) with that x;
//   4. B (the Toeplitz bands of the warp's 4 channels) stays in registers for
//      all units of a channel tile;
//   5. the results, rounded to 16 bits, go to a separate 64B-swizzled NHWC
//      output tile and leave with one TMA tensor store (clipped at the
//      tensor edges by the copy engine).
// Two CTA barriers per unit: "T and the output tile are ready" and "the
// output tile is complete (and every warp is done with T)".
#pragma once

#include "mma_common.cuh"

namespace dwc {
namespace {

using namespace tiled;
using namespace mma;

#ifndef DWCONV_MMA
#define DWCONV_MMA 1  // 0: leave every shape to the CUDA-core kernels
#endif

#ifndef DWCONV_MMA_CHAIN_G
#define DWCONV_MMA_CHAIN_G 4  // largest G whose operands are loaded in chains (half of each from registers)
#endif

constexpr int kCh = 32;                 // channels per work unit
constexpr int kChPerWarp = 4;           // channels per warp
constexpr int kMThreads = kCh / kChPerWarp * 32;
constexpr int kPB = 2 * kCh;            // bytes of one staged pixel (= swizzle span)

// Shared-memory address of a byte offset inside a buffer with the TMA's
// 64-byte swizzle (16-byte chunk bits 4-5 XOR address bits 7-8).
__device__ __forceinline__ unsigned swz(unsigned a) { return a ^ (((a >> 7) & 3u) << 4); }

// Tile geometry, fixed by the filter height, G, the images per unit NI and
// the row sets per unit KNB; ES = bytes of a staged input element (2, or 1
// for FP8 inputs, whose halo is converted to f16 during the transposition).
template <int FH, int G, int NI, int KNB, int ES = 2>
struct Cfg {
    static constexpr int RB = 8 / G;                              // output rows of an 8-row M block
    static constexpr int OTH = NI == 1 ? 2 * KNB * RB : KNB * RB; // output rows per image
    static constexpr int OTW = 8 * G;                             // output columns
    static constexpr int HRI = OTH + FH - 1;                      // staged rows per image
    static constexpr int DHT = NI == 1 ? KNB * RB : HRI;          // T rows from M rows 0-7 to 8-15
    static constexpr int OHB = NI == 1 ? KNB * RB : OTH;          // output-tile rows, same
    static constexpr int TR = NI * HRI, SW = OTW + 8;             // staged rows, columns
    static constexpr int RS = SW;                                 // T row stride (halves)
    static constexpr int CS = channel_stride(TR * RS);            // T channel stride (halves)
    // Row set j covers output rows base(j) + G i, i < RB (and the same rows
    // OHB lower for M rows 8-15); the KNB sets tile the rows exactly when KNB
    // is a multiple of G (or G = 8, one row per block).
    __host__ __device__ static constexpr int base(int j) { return j % G + 8 * (j / G); }
    static constexpr int NQ = base(KNB - 1) + FH;                 // A operands per channel
    static constexpr unsigned s_bytes = TR * SW * kCh * ES;
    static constexpr unsigned s_stride = align1k(s_bytes);
    static constexpr unsigned t_bytes = align1k(kCh * CS * 2);
    static constexpr unsigned o_bytes = NI * OTH * OTW * kPB;
    static constexpr int NS = 2 * s_stride + t_bytes + o_bytes + 1024 <= 227 * 1024 ? 2 : 1;  // staging buffers
    static constexpr unsigned t_off = NS * s_stride;
    static constexpr unsigned o_off = t_off + t_bytes;
    static constexpr unsigned smem = o_off + o_bytes;             // + 1 KB alignment slack at launch
    static constexpr int MINB = smem + 2048 <= 113 * 1024 ? 2 : 1;  // CTAs per SM registers are capped for
};

// FUSE: the BN+Act prologue and affine+activation epilogue of the fused
// forward pass are compiled in (a separate instance, so that the plain
// passes keep their own register allocation).
template <typename T> __host__ __device__ constexpr int in_es() { return sizeof(T) == 1 ? 1 : 2; }

// Input element to tensor-core operand type (exact for every supported pair).
template <typename TM, typename T>
__device__ __forceinline__ TM to_operand(T v) {
    if constexpr (std::is_same<T, TM>::value)
        return v;
    else
        return from_f32<TM>(to_f32(v));
}

template <typename T, int FH, int FW, int G, int NI, int KNB, bool FUSE>
__global__ void __launch_bounds__(kMThreads, (Cfg<FH, G, NI, KNB, in_es<T>()>::MINB))
    tiled_mma_kernel(const __grid_constant__ CUtensorMap halo_map, const __grid_constant__ CUtensorMap out_map,
                     TiledConv p, GeoM g, unsigned *err) {
    using C = Cfg<FH, G, NI, KNB, in_es<T>()>;
    constexpr int DHT = C::DHT, NQ = C::NQ, NS = C::NS;
    static_assert(G == 8 || KNB % G == 0, "row sets must tile the unit's rows");
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    __shared__ __align__(8) uint64_t bar[NS];
    using TM = typename MmaIn<T>::type;   // MMA operand type
    using TO = typename OutOf<T>::type;   // output type
    using Op = MmaOp<TM>;

    // Swizzled buffers start on 1024-byte boundaries (the launch adds 1 KB of slack).
    unsigned char *smem_raw = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int gq = lane / 4, t4 = lane % 4;  // mma fragment coordinates
    unsigned char *S = smem_raw;             // NS staging buffers [NI][HRI][SW][32], s_stride apart
    const unsigned s_addr = smem_addr(S);
    const unsigned t_addr = s_addr + C::t_off;  // T [32][CS] halves
    const unsigned o_addr = s_addr + C::o_off;  // output tile [NI][OTH][OTW][32], swizzled
    const T *wg = static_cast<const T *>(p.w);

    // Contiguous unit range of this CTA (channel tile slowest: few B reloads).
    const int u_begin = (int)((long long)g.units * blockIdx.x / gridDim.x);
    const int u_end = (int)((long long)g.units * (blockIdx.x + 1) / gridDim.x);

    if (tid == 0) {
        for (int b = 0; b < NS; ++b) mbar_init(&bar[b], 1);
        mbar_fence_init();
    }
    __syncthreads();

    // Unit cursors (row band fastest) for the loads (thread 0) and the compute.
    Unit ld = decode(g, u_begin), cur = ld;
    auto issue = [&](int b) {
        const Unit un = ld;
        advance(g, g.groups, ld);
        mbar_arrive_expect_tx(&bar[b], C::s_bytes);
        tma_load_4d(S + b * C::s_stride, &halo_map, un.ctile * kCh, un.twi * C::OTW - p.pad_w,
                    un.band * C::OTH - p.pad_h, un.group * NI, &bar[b]);
    };
    if (tid == 0)
        for (int b = 0; b < NS && u_begin + b < u_end; ++b) issue(b);

    // A operand x of a channel = one ldmatrix.x4: matrix j (lanes 8j..8j+7
    // give its row addresses) holds M rows 8(j%2)..+7 and k 8(j/2)..+7; M row
    // i of block j%2 is window i % G of T row x + G (i / G) + DHT (j%2).
    const int mj = lane / 8, mi = lane % 8;
    const int lane_off = ((mj & 1) * DHT + (mi / G) * G) * C::RS + 8 * (mi % G) + 8 * (mj >> 1);
    // ldmatrix.x2 of T rows x + DHT alone: matrix mj & 1 = k half.
    const int lane_off2 = (DHT + (mi / G) * G) * C::RS + 8 * (mi % G) + 8 * (mj & 1);
    // Transposition: one ldmatrix.x4 = the 4 16-byte channel chunks of 8
    // pixels; this lane addresses row tr of matrix tj.
    const int tr = lane % 8, tj = lane / 8;
    // Output: lane (gq, t4) writes position (row G (gq / G) (+ OHB for M rows
    // 8-15), column 8 (gq % G) + 2t4 + e) of each row set; the bits the
    // swizzle reads (7 and up) do not depend on the row set or on e, so the
    // lane's swizzled chunk is fixed.
    const unsigned o_pos = (unsigned)((gq / G) * G * C::OTW + 8 * (gq % G) + 2 * t4) * kPB;
    const unsigned o_lane = o_addr + swz(o_pos + (unsigned)warp * 8);
    const unsigned o_lane0 = o_lane + (gq & 1) * kPB, o_lane1 = o_lane + (1 - (gq & 1)) * kPB;

    int loaded_ctile = -1;
    float bias_r[kChPerWarp];
    unsigned bfr[kChPerWarp][FH][2];  // Toeplitz bands, B fragments (k 0-7, k 8-15)
    for (int u = u_begin, k = 0; u < u_end; ++u, ++k, advance(g, g.groups, cur)) {
        if (cur.ctile != loaded_ctile) {
            // B[k][n] = w[fh][k - n]: lane (gq, t4) holds k = 2t4, 2t4+1 (+8), n = gq.
            // For the input gradient the filter is rotated by 180 degrees.
            loaded_ctile = cur.ctile;
            const int cc0 = cur.ctile * kCh + warp * kChPerWarp;
#pragma unroll
            for (int ci = 0; ci < kChPerWarp; ++ci) {
                const int cc = cc0 + ci;
                bias_r[ci] = (p.bias && cc < p.C) ? p.bias[cc] : 0.f;
            }
            if constexpr (sizeof(T) == 2 && std::is_same<T, TM>::value && G < 8) {
                // 16-bit filters on maps of at most 32 columns (few units per
                // channel tile and CTA): the warp's 4 channels of a tap are one
                // 8-byte word, read with one load where it is aligned and
                // complete (C a multiple of 4), else half by half, with the
                // loads of 4 filter rows in flight together.  Measured on
                // GB300: 14x14 maps 9 % and 28x28 maps 2-4 % faster; at G = 8
                // (one reload per ~18 units) the per-channel loads below keep a
                // register allocation that is 4 % faster.
                const bool vec = p.C % kChPerWarp == 0 && cc0 + kChPerWarp <= p.C &&
                                 (reinterpret_cast<uintptr_t>(wg) & 7u) == 0;
                const unsigned short *wh = reinterpret_cast<const unsigned short *>(wg);
#pragma unroll
                for (int fh = 0; fh < FH; ++fh) {
                    const int sfh = p.flip ? FH - 1 - fh : fh;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint2 q[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int fw = 2 * t4 + e + 8 * h - gq;
                            q[e] = make_uint2(0u, 0u);
                            if (fw < 0 || fw >= FW) continue;
                            const size_t at = (size_t)(sfh * FW + (p.flip ? FW - 1 - fw : fw)) * p.C + cc0;
                            if (vec) {
                                q[e] = __ldg(reinterpret_cast<const uint2 *>(wh + at));
                            } else {
                                unsigned hv[kChPerWarp];
#pragma unroll
                                for (int ci = 0; ci < kChPerWarp; ++ci)
                                    hv[ci] = cc0 + ci < p.C ? (unsigned)__ldg(wh + at + ci) : 0u;
                                q[e] = make_uint2(hv[0] | (hv[1] << 16), hv[2] | (hv[3] << 16));
                            }
                        }
                        // Channel ci is half ci % 2 of word ci / 2; B pair (e = 0, 1).
                        bfr[0][fh][h] = __byte_perm(q[0].x, q[1].x, 0x5410);
                        bfr[1][fh][h] = __byte_perm(q[0].x, q[1].x, 0x7632);
                        bfr[2][fh][h] = __byte_perm(q[0].y, q[1].y, 0x5410);
                        bfr[3][fh][h] = __byte_perm(q[0].y, q[1].y, 0x7632);
                    }
                    if (fh % 4 == 3) asm volatile("" ::: "memory");  // 4 rows of loads at a time
                }
            } else {
#pragma unroll
                for (int ci = 0; ci < kChPerWarp; ++ci) {
                    const int cc = cc0 + ci;
                    const bool live = cc < p.C;
#pragma unroll
                    for (int fh = 0; fh < FH; ++fh) {
                        const int sfh = p.flip ? FH - 1 - fh : fh;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            TM v[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int fw = 2 * t4 + e + 8 * h - gq;
                                v[e] = from_f32<TM>(0.f);
                                if (live && fw >= 0 && fw < FW)
                                    v[e] = to_operand<TM>(wg[(sfh * FW + (p.flip ? FW - 1 - fw : fw)) * p.C + cc]);
                            }
                            bfr[ci][fh][h] = Op::pack_raw(v[0], v[1]);
                        }
                    }
                }
            }
        }
        if (!mbar_wait(&bar[k % NS], (k / NS) & 1)) {
            // Give up on this unit; thread 0 lets its copies in flight end
            // (again with bounded waits) before the CTA leaves.
            report_timeout(err);
            if (tid == 0) {
                for (int j = k; j < k + NS && u_begin + j < u_end; ++j) mbar_wait(&bar[j % NS], (j / NS) & 1);
                asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
            }
            return;
        }

        // Transpose S[row][col][ch] -> T[ch][row][col], 8 columns x 32
        // channels per step: ldmatrix.trans gives lane (gq, t4) cols 2t4,
        // 2t4+1 of channel 8 chunk + gq; stmatrix writes them as the 16-byte
        // row (channel, row, 8 cols).  Every warp finished reading T (previous
        // unit) before the last barrier.
        const unsigned s_buf = s_addr + (k % NS) * C::s_stride;
        // With a BN+Act prologue (Flash-DWC §5.2) every staged value passes
        // through registers here anyway: lane (gq, t4) holds channel
        // 8 tj + gq of columns col0 + 2t4, +1 in register tj; positions
        // outside the input are padding of x' and stay zero.
        auto transpose = [&](auto pre) {
            constexpr int PA = decltype(pre)::value;  // activation, or -1: no prologue
            float2 s2[4], t2[4];
            unsigned cmask = 0;  // bit 2i + e: column 8i + 2t4 + e lies inside the input
            if constexpr (PA >= 0) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = cur.ctile * kCh + 8 * m + gq;
                    const Affine a = c < p.C ? affine_in(p.fz, c) : Affine{1.f, 0.f};
                    s2[m] = make_float2(a.s, a.s);
                    t2[m] = make_float2(a.t, a.t);
                }
                const int iw0 = cur.twi * C::OTW - p.pad_w + 2 * t4;
#pragma unroll
                for (int i = 0; i < C::SW / 8; ++i)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int iw = iw0 + 8 * i + e;
                        cmask |= (iw >= 0 && iw < p.Ws ? 1u : 0u) << (2 * i + e);
                    }
            }
            const int ih0 = cur.band * C::OTH - p.pad_h;
            constexpr int kSteps = C::TR * (C::SW / 8), kStride = kMThreads / 32;
            auto src = [&](int b) {
                const int row = b / (C::SW / 8), col0 = (b % (C::SW / 8)) * 8;
                return s_buf + swz((unsigned)((row * C::SW + col0 + tr) * kPB + 16 * tj));
            };
            auto dst = [&](int b) {
                const int row = b / (C::SW / 8), col0 = (b % (C::SW / 8)) * 8;
                return t_addr + 2u * ((8 * tj + tr) * C::CS + row * C::RS + col0);
            };
            if constexpr (sizeof(T) == 1) {
                // FP8: the staged pixel is 32 bytes, unswizzled.  Lane (gq, t4)
                // gathers channel 8m + gq of columns col0 + 2t4, +1 -- the
                // layout ldmatrix.trans gives for 16-bit data -- and converts
                // each pair exactly to f16.
                const unsigned char *s8 = smem_raw + (k % NS) * C::s_stride;
                auto gather = [&](int b, unsigned (&v)[4]) {
                    const int row = b / (C::SW / 8), col0 = (b % (C::SW / 8)) * 8;
                    const unsigned char *px = s8 + (row * C::SW + col0 + 2 * t4) * kCh + gq;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const __nv_fp8x2_storage_t pr =
                            (__nv_fp8x2_storage_t)(px[8 * m] | ((unsigned)px[kCh + 8 * m] << 8));
                        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
                        v[m] = *reinterpret_cast<const unsigned *>(&h);
                    }
                };
                // Two steps per iteration: both gathers before the stores.
                int b = warp;
                for (; b + kStride < kSteps; b += 2 * kStride) {
                    unsigned v[2][4];
                    gather(b, v[0]);
                    gather(b + kStride, v[1]);
                    stsm_x4(dst(b), v[0][0], v[0][1], v[0][2], v[0][3]);
                    stsm_x4(dst(b + kStride), v[1][0], v[1][1], v[1][2], v[1][3]);
                }
                for (; b < kSteps; b += kStride) {
                    unsigned v[4];
                    gather(b, v);
                    stsm_x4(dst(b), v[0], v[1], v[2], v[3]);
                }
            } else if constexpr (PA < 0) {
                // Two steps per iteration: both loads are in flight before the
                // stores (measured on GB300: 4 % faster fwd/dgrad at 7x7).
                int b = warp;
                for (; b + kStride < kSteps; b += 2 * kStride) {
                    unsigned v[2][4];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        ldsm_x4_trans(v[u][0], v[u][1], v[u][2], v[u][3], src(b + u * kStride));
#pragma unroll
                    for (int u = 0; u < 2; ++u) stsm_x4(dst(b + u * kStride), v[u][0], v[u][1], v[u][2], v[u][3]);
                }
                for (; b < kSteps; b += kStride) {
                    unsigned v[4];
                    ldsm_x4_trans(v[0], v[1], v[2], v[3], src(b));
                    stsm_x4(dst(b), v[0], v[1], v[2], v[3]);
                }
            } else {
                // Two steps per iteration as in the plain transposition (measured
                // on GB300: 5 % faster with a ReLU prologue; issuing the next
                // step's load before this step's arithmetic, or skipping
                // all-padding steps, was slower).
                auto keep_of = [&](int b) {
                    const int row = b / (C::SW / 8), chunk = b % (C::SW / 8);
                    const int img = row / C::HRI, ih = ih0 + row - img * C::HRI;
                    const bool rok = ih >= 0 && ih < p.Hs && cur.group * NI + img < p.N;
                    const unsigned m2 = rok ? (cmask >> (2 * chunk)) & 3u : 0u;
                    return (m2 & 1u ? 0x0000FFFFu : 0u) | (m2 & 2u ? 0xFFFF0000u : 0u);
                };
                int b = warp;
                for (; b + kStride < kSteps; b += 2 * kStride) {
                    unsigned v[2][4];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        ldsm_x4_trans(v[u][0], v[u][1], v[u][2], v[u][3], src(b + u * kStride));
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const unsigned keep = keep_of(b + u * kStride);
#pragma unroll
                        for (int m = 0; m < 4; ++m) v[u][m] = prologue_packed<T, PA>(v[u][m], s2[m], t2[m]) & keep;
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) stsm_x4(dst(b + u * kStride), v[u][0], v[u][1], v[u][2], v[u][3]);
                }
                for (; b < kSteps; b += kStride) {
                    unsigned v[4];
                    ldsm_x4_trans(v[0], v[1], v[2], v[3], src(b));
                    const unsigned keep = keep_of(b);
#pragma unroll
                    for (int m = 0; m < 4; ++m) v[m] = prologue_packed<T, PA>(v[m], s2[m], t2[m]) & keep;
                    stsm_x4(dst(b), v[0], v[1], v[2], v[3]);
                }
            }
        };
        if (FUSE && p.fz.pre())
            with_act(p.fz.in_act, transpose);
        else
            transpose(std::integral_constant<int, -1>{});
        // The previous unit's TMA store must have read the output tile.
        if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
        __syncthreads();  // T ready, output tile free, this staging buffer free
        if (tid == 0 && u + NS < u_end) issue(k % NS);

        // MMAs.  Each step loads the next operand (also across channels)
        // and runs the MMAs of the current one, row sets interleaved
        // (independent accumulators).  With one image per unit the upper half
        // of operand x (T rows x + DHT) is the lower half of operand x + DHT,
        // so the operands of a channel are taken in chains x = r, r + DHT,
        // r + 2 DHT, ...: a chain's first operand is one ldmatrix.x4, every
        // later one copies its lower half from registers and loads only its
        // upper half (one ldmatrix.x2).  Measured on GB300 (bf16 7x7
        // training layers): a small gain at G = 4 (28x28 maps, forward + dgrad
        // 0.068 against 0.069 ms), a loss at G = 8 (56x56, forward 0.050
        // against 0.049 ms), so chains are used for G <= DWCONV_MMA_CHAIN_G.  The order of the
        // MMAs on an accumulator is fixed at compile time, so results do not
        // vary from call to call.
        float d[kChPerWarp][KNB][4];
        constexpr bool kChain = NI == 1 && G <= DWCONV_MMA_CHAIN_G;
        constexpr int NR = kChain ? (DHT < NQ ? DHT : NQ) : 1;  // chains per channel
        constexpr int XS = kChain ? DHT : 1;                      // operand step within a chain
        auto op_addr = [&](int ci, int x) { return t_addr + 2u * ((warp * kChPerWarp + ci) * C::CS + x * C::RS); };
        unsigned a[4], an[4];
        ldsm_x4(a[0], a[1], a[2], a[3], op_addr(0, 0) + 2u * lane_off);
#pragma unroll
        for (int ci = 0; ci < kChPerWarp; ++ci) {
#pragma unroll
            for (int j = 0; j < KNB; ++j) d[ci][j][0] = d[ci][j][1] = d[ci][j][2] = d[ci][j][3] = bias_r[ci];
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int x = r; x < NQ; x += XS) {
                    bool next = true;
                    if (x + XS < NQ) {
                        if constexpr (kChain) {
                            an[0] = a[1];
                            an[2] = a[3];
                            ldsm_x2(an[1], an[3], op_addr(ci, x + XS) + 2u * lane_off2);
                        } else {
                            ldsm_x4(an[0], an[1], an[2], an[3], op_addr(ci, x + 1) + 2u * lane_off);
                        }
                    } else if (r + 1 < NR) {
                        ldsm_x4(an[0], an[1], an[2], an[3], op_addr(ci, r + 1) + 2u * lane_off);
                    } else if (ci + 1 < kChPerWarp) {
                        ldsm_x4(an[0], an[1], an[2], an[3], op_addr(ci + 1, 0) + 2u * lane_off);
                    } else {
                        next = false;
                    }
#pragma unroll
                    for (int j = 0; j < KNB; ++j) {
                        const int fh = x - C::base(j);
                        if (fh >= 0 && fh < FH)
                            Op::run(d[ci][j], a[0], a[1], a[2], a[3], bfr[ci][fh][0], bfr[ci][fh][1]);
                    }
                    if (next)
#pragma unroll
                        for (int e = 0; e < 4; ++e) a[e] = an[e];
                }
        }

        // Epilogue of the fused forward pass: per-channel affine map and
        // activation on the fp32 sums, before the rounding.
        if (FUSE && p.fz.post())
            with_act(p.fz.out_act, [&](auto act) {
#pragma unroll
                for (int ci = 0; ci < kChPerWarp; ++ci) {
                    const int cc = cur.ctile * kCh + warp * kChPerWarp + ci;
                    const Affine a = cc < p.C ? affine_out(p.fz, cc) : Affine{1.f, 0.f};
#pragma unroll
                    for (int j = 0; j < KNB; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            d[ci][j][e] = activate(fmaf(a.s, d[ci][j][e], a.t), decltype(act)::value);
                }
            });

        // Output tile, 64B-swizzled for the TMA store: this lane writes 8
        // bytes (its warp's 4 channels) per output position.  The two columns
        // 2t4, 2t4+1 go out in the order set by gq's parity, so one store
        // covers both 64-byte halves of a 128-byte line (4-way instead of
        // 8-way bank conflicts).
#pragma unroll
        for (int j = 0; j < KNB; ++j)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                unsigned lo[2], hi[2];  // column 2t4 + e: channels (0, 1), (2, 3)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    lo[e] = MmaOp<TO>::pack(d[0][j][2 * half + e], d[1][j][2 * half + e]);
                    hi[e] = MmaOp<TO>::pack(d[2][j][2 * half + e], d[3][j][2 * half + e]);
                }
                const bool odd = gq & 1;
                const unsigned row = (C::base(j) + half * C::OHB) * C::OTW * kPB;
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};\n" ::"r"(o_lane0 + row), "r"(odd ? lo[1] : lo[0]),
                             "r"(odd ? hi[1] : hi[0])
                             : "memory");
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};\n" ::"r"(o_lane1 + row), "r"(odd ? lo[0] : lo[1]),
                             "r"(odd ? hi[0] : hi[1])
                             : "memory");
            }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // visible to the TMA store
        __syncthreads();  // output tile complete; every warp is done with T
        if (tid == 0) {
            asm volatile(
                "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];\n" ::"l"(
                    reinterpret_cast<uint64_t>(&out_map)),
                "r"(cur.ctile * kCh), "r"(cur.twi * C::OTW), "r"(cur.band * C::OTH), "r"(cur.group * NI),
                "r"(o_addr)
                : "memory");
            asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
        }
    }
    if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}

// Halo map as for the CUDA-core kernels (box: 32 channels x columns x rows x
// images), with the 64-byte swizzle for 16-bit data (the inner box row is
// exactly one 32-channel pixel).
inline bool make_mma_halo_map(CUtensorMap *map, const TiledConv &p, dwconv_dtype dt, size_t es, const uint32_t box[4],
                              int swizzle) {
    const char *base = static_cast<const char *>(p.in) + ((size_t)p.in_off_h * p.Wf + p.in_off_w) * p.C * es;
    const uint64_t dims[4] = {(uint64_t)p.C, (uint64_t)p.Ws, (uint64_t)p.Hs, (uint64_t)p.N};
    const uint64_t str[3] = {(uint64_t)p.in_step_w * p.C * es, (uint64_t)p.in_step_h * p.Wf * p.C * es,
                             (uint64_t)p.Hf * p.Wf * p.C * es};
    return encode_tmap_4d(map, dt, base, dims, str, box, swizzle);
}

template <typename T, int FH, int FW, int G, int NI, int KNB, bool FUSE>
cudaError_t run(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    using C = Cfg<FH, G, NI, KNB, in_es<T>()>;
    if (C::smem + 1024 > 227 * 1024) return cudaErrorNotSupported;
    GeoM g{};
    g.tiles_h = (p.OHs + C::OTH - 1) / C::OTH;
    g.tiles_w = (p.OWs + C::OTW - 1) / C::OTW;
    g.groups = (p.N + NI - 1) / NI;
    const long long per = (long long)g.groups * g.tiles_w * g.tiles_h;
    const long long units = per * ((p.C + kCh - 1) / kCh);
    if (units >= (1LL << 30)) return cudaErrorNotSupported;
    g.per_ctile = (int)per;
    g.units = (int)units;
    // The output map covers y (or dx) directly; the TMA store clips the tile
    // at the edges.
    const uint32_t box[4] = {(uint32_t)kCh, (uint32_t)C::SW, (uint32_t)C::HRI, (uint32_t)NI};
    const uint32_t obox[4] = {(uint32_t)kCh, (uint32_t)C::OTW, (uint32_t)C::OTH, (uint32_t)NI};
    CUtensorMap map, omap;
    // FP8: the halo is staged unswizzled (32-byte pixels) and gathered bytewise;
    // the output is bf16.
    const dwconv_dtype out_dt = dt == DWCONV_FP8_E4M3 ? DWCONV_BF16 : dt;
    if (!make_mma_halo_map(&map, p, dt, sizeof(T), box, sizeof(T) == 1 ? 0 : kPB) ||
        !make_out_map(&omap, p, out_dt, sizeof(typename OutOf<T>::type), obox, kPB))
        return cudaErrorNotSupported;
    auto kern = tiled_mma_kernel<T, FH, FW, G, NI, KNB, FUSE>;
    int per_sm = 0;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kMThreads, C::smem + 1024, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const long long slots = (long long)sm_count() * per_sm;
    const int grid = (int)std::min<long long>(g.units, slots);
    kern<<<grid, kMThreads, C::smem + 1024, st>>>(map, omap, p, g, device_error_word());
    note_launches(1);
    note_kernel("tiled_mma");
    return cudaGetLastError();
}

// Tile shape by map width: one image and 8 groups of 8 columns per M block
// down to two images and 2 groups of 4 rows.  Maps of at most 8 columns stay
// on the CUDA-core kernel: with 8-row units of two images (G = 1) a unit has
// only FH MMAs per channel and the transposition and barriers dominate
// (measured on GB300, bf16 7x7 on 7x7 maps: 0.033 ms against 0.024 ms).
template <typename T, int FH, int FW, bool FUSE>
cudaError_t by_width(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (p.OWs > 32) return run<T, FH, FW, 8, 1, 4, FUSE>(p, dt, st);
    if (p.OWs > 16) return run<T, FH, FW, 4, 1, 4, FUSE>(p, dt, st);
    if (p.OWs > 8) return run<T, FH, FW, 2, 2, 4, FUSE>(p, dt, st);
    return cudaErrorNotSupported;
}

template <typename T, bool FUSE>
cudaError_t by_filter(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (p.FH == 7 && p.FW == 7) return by_width<T, 7, 7, FUSE>(p, dt, st);
    if (p.FH == 5 && p.FW == 5) return by_width<T, 5, 5, FUSE>(p, dt, st);
    if (p.FH == 3 && p.FW == 3) return by_width<T, 3, 3, FUSE>(p, dt, st);
    return cudaErrorNotSupported;
}

}  // namespace

}  // namespace dwc
