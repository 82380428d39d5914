// Warp-specialised tensor-core forward pass and stride-1 input gradient for
// 16-bit data, 5x5 and 7x7 filters and maps wider than 32 columns (the kernel
// also compiles for 3x3).
//
// The arithmetic is that of tiled_mma_kernel.cuh at G = 8 (Flash-DWC §4.2
// Toeplitz packing: one mma.sync m16n8k16 takes the 8 groups of 8 columns of
// one output row in M rows 0-7 and of the row 4 below in M rows 8-15; a unit
// is 8 output rows x 64 columns x 32 channels, four row sets).  What changes
// is how the input reaches the MMAs:
//
//   - A column of units (one image, one 64-column strip, one channel tile) is
//     read as pieces of 8 input rows: piece i holds input rows 8i - pad_h to
//     8i + 7 - pad_h.  The unit of output rows 8b .. 8b + 7 reads all of
//     piece b and the first FH - 1 rows of piece b + 1, so a unit below the
//     previous one needs one new piece: each input row is copied from L2 and
//     transposed once per column instead of (8 + FH - 1) / 8 times.
//   - Warpgroup 0 (warps 0-3) is the producer: thread 0 issues the TMA copy of
//     each piece (zero-filled outside the input) into one of two staging
//     slots, and the four warps transpose each staged piece (ldmatrix.trans +
//     stmatrix) into its slot of a three-piece channel-major ring
//     T[channel][24 rows][72 columns].
//   - Warpgroups 1-2 (warps 4-11, 4 channels each) are the consumers: the
//     MMAs of a unit read its 8 + FH - 1 rows from two consecutive ring slots
//     (the row index wraps at 24) while the producer fills the third, then
//     they round the sums to 16 bits into the output tile, which one thread
//     sends out with a TMA store.
//
// The producer needs few registers and the MMA warps many (accumulators and
// the Toeplitz bands of their 4 channels): setmaxnreg moves them, 56 per
// producer thread and 224 per consumer thread out of the 384 x 168 the CTA is
// launched with.
//
// Synchronisation: mbarriers between the roles (staging slot full: TMA
// transaction bytes; ring slot full: one arrival per producer warp; ring slot
// free: one arrival per consumer warp), named barriers inside each role (the
// producer's staging slot is free once all four warps have read it; the
// consumers' output tile is free, then complete).  Every wait is bounded; a
// wait that runs out sets the device error word and a CTA-wide flag after
// which no role waits any more, so every thread still reaches the end of its
// loop and every named barrier.
#pragma once

#include <atomic>

#include "tiled_mma_kernel.cuh"

namespace dwc {
namespace {

#ifndef DWCONV_MMA_RING
#define DWCONV_MMA_RING 1  // 0: maps wider than 32 columns use tiled_mma_kernel at G = 8
#endif
#ifndef DWCONV_RING_CHAIN
#define DWCONV_RING_CHAIN 1  // A operands in chains (upper half of x = lower half of x + DHT)
#endif
#ifndef DWCONV_RING_SPLIT
#define DWCONV_RING_SPLIT 0  // 1: the two consumer warpgroups run independently (16 channels each)
#endif

struct CfgR {
    static constexpr int PR = 8;                 // rows of a piece = output rows of a unit
    static constexpr int OTW = 64, SW = 72;      // output columns, staged columns
    static constexpr int DHT = 4;                // T rows from M rows 0-7 to M rows 8-15
    static constexpr int KNB = 4;                // row sets per unit
    static constexpr int NSLOT = 3, NSTAGE = 2;  // ring slots, staging slots
    static constexpr int TRR = NSLOT * PR;       // ring rows
    static constexpr int RS = SW;                // T row stride (halves)
    static constexpr int CS = channel_stride(TRR * RS);  // T channel stride (halves), 8 mod 16
    static constexpr unsigned s_bytes = PR * SW * kPB;   // one staged piece, 64-byte swizzled
    static constexpr unsigned t_off = NSTAGE * s_bytes;
    static constexpr unsigned t_bytes = align1k(kCh * CS * 2);
    static constexpr unsigned o_off = t_off + t_bytes;
    static constexpr unsigned o_bytes = PR * OTW * kPB;  // output tile [8][64][32] (or two [8][64][16]), swizzled
    static constexpr unsigned f_off = o_off + o_bytes;   // filter slab [FH FW][32] halves, FH FW <= 49
    static constexpr unsigned f_bytes = (49 * kCh * 2 + 127u) & ~127u;
    static constexpr unsigned smem = f_off + f_bytes;    // + 1 KB alignment slack at launch
    static constexpr int kGroups = DWCONV_RING_SPLIT ? 2 : 1;  // independent consumer groups
    static constexpr int kThreads = 384, kProdThreads = 128;
    static constexpr int kProdRegs = 56, kMmaRegs = 224, kLaunchRegs = 168;
};
static_assert(CfgR::s_bytes % 1024 == 0 && CfgR::t_off % 1024 == 0 && CfgR::o_off % 1024 == 0,
              "swizzled buffers start on 1024-byte boundaries");
static_assert(CfgR::smem + 1024 <= 227 * 1024, "shared memory of one CTA");
static_assert(CfgR::kProdThreads * CfgR::kProdRegs + (CfgR::kThreads - CfgR::kProdThreads) * CfgR::kMmaRegs <=
                  CfgR::kThreads * CfgR::kLaunchRegs,
              "the register split must fit in the registers the CTA is launched with");
static_assert(CfgR::kLaunchRegs * CfgR::kThreads <= 65536, "one CTA per SM");

// Bounded mbarrier wait that also gives up as soon as another thread of the
// CTA has given up (*abort set); a wait that runs out sets *abort and the
// device error word.  Returns false if it did not see the phase complete.
__device__ __forceinline__ bool ring_wait(uint64_t *bar, unsigned parity, volatile int *abort, unsigned *err) {
    if (*abort) return false;
    const unsigned a = smem_addr(bar);
    for (unsigned i = 0; i < kSpinLimit; ++i) {
        unsigned done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 1023u) == 1023u && *abort) return false;
    }
    *abort = 1;
    report_timeout(err);
    return false;
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

template <typename T, int FH, int FW>
__global__ void __launch_bounds__(CfgR::kThreads, 1)
    tiled_mma_ring_kernel(const __grid_constant__ CUtensorMap halo_map, const __grid_constant__ CUtensorMap out_map,
                          TiledConv p, GeoM g, unsigned *err) {
    using C = CfgR;
    constexpr int NQ = (C::KNB - 1) + FH;  // A operands per channel: row sets 0-3 start at rows 0-3
    static_assert(FH - 1 <= C::PR, "a unit reads at most two pieces");
    static_assert(FH * FW <= 49, "filter slab");
    static_assert(NQ - 1 + C::DHT < C::PR + C::PR, "a unit's rows lie in two ring slots");
    extern __shared__ __align__(1024) unsigned char smem_dyn[];
    __shared__ __align__(8) uint64_t sfull[C::NSTAGE], tfull[C::NSLOT], tempty[C::NSLOT];
    __shared__ int abort_flag;
    volatile int *abort = &abort_flag;
    using Op = MmaOp<T>;

    unsigned char *S = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    const unsigned s_addr = smem_addr(S);
    const unsigned t_addr = s_addr + C::t_off;  // T [32][CS] halves: 3 slots of 8 rows x 72 columns
    const unsigned o_addr = s_addr + C::o_off;  // output tile [8][64][32], swizzled
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    // Contiguous unit range of this CTA (row band fastest, channel tile slowest).
    const int u_begin = (int)((long long)g.units * blockIdx.x / gridDim.x);
    const int u_end = (int)((long long)g.units * (blockIdx.x + 1) / gridDim.x);
    // Pieces of the range: one per unit, plus one for the first unit and for
    // every later unit that starts a column (band 0: unit index % tiles_h == 0).
    const int n_pieces =
        u_end > u_begin ? (u_end - u_begin) + 1 + ((u_end - 1) / g.tiles_h - u_begin / g.tiles_h) : 0;

    if (tid == 0) {
        for (int b = 0; b < C::NSTAGE; ++b) mbar_init(&sfull[b], 1);
        for (int b = 0; b < C::NSLOT; ++b) {
            mbar_init(&tfull[b], C::kProdThreads / 32);
            mbar_init(&tempty[b], (C::kThreads - C::kProdThreads) / 32);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (n_pieces == 0) return;

    if (warp < C::kProdThreads / 32) {
        // ---------------- producer: TMA copies and transposition ----------------
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(C::kProdRegs));
        // Copy cursor (thread 0): the unit whose piece comes next, and whether
        // the first of a two-piece (column-starting) unit has been issued.
        Unit lu = decode(g, u_begin);
        bool lfirst = true, lsecond = false;
        int issued = 0;
        auto issue = [&]() {
            const Unit un = lu;
            int prow;
            if ((lfirst || un.band == 0) && !lsecond) {
                prow = un.band;
                lsecond = true;
            } else {
                prow = un.band + 1;
                lsecond = false;
                lfirst = false;
                advance(g, g.groups, lu);
            }
            uint64_t *b = &sfull[issued % C::NSTAGE];
            mbar_arrive_expect_tx(b, C::s_bytes);
            tma_load_4d(S + (issued % C::NSTAGE) * C::s_bytes, &halo_map, un.ctile * kCh, un.twi * C::OTW - p.pad_w,
                        prow * C::PR - p.pad_h, un.group, b);
            ++issued;
        };
        if (tid == 0)
            for (int j = 0; j < C::NSTAGE && j < n_pieces; ++j) issue();

        // Transposition of a piece, 8 columns x 32 channels per step:
        // ldmatrix.trans gives lane (gq, t4) columns 2t4, 2t4+1 of channel
        // 8 chunk + gq; stmatrix writes them as the 16-byte row (channel, row,
        // 8 columns) of T.  72 steps, 18 per warp, two in flight.
        const int tr = lane % 8, tj = lane / 8;
        constexpr int kChunks = C::SW / 8, kSteps = C::PR * kChunks, kStride = C::kProdThreads / 32;
        static_assert(kSteps % (2 * kStride) == 0, "whole double steps per warp");
        for (int j = 0; j < n_pieces; ++j) {
            const int slot = j % C::NSLOT, ss = j % C::NSTAGE;
            if (j >= C::NSLOT) ring_wait(&tempty[slot], (unsigned)((j / C::NSLOT) - 1) & 1u, abort, err);
            ring_wait(&sfull[ss], (unsigned)(j / C::NSTAGE) & 1u, abort, err);
            const unsigned s_buf = s_addr + ss * C::s_bytes;
            const unsigned t_slot = t_addr + 2u * (unsigned)(slot * C::PR * C::RS);
            auto src = [&](int b) {
                const int row = b / kChunks, col0 = (b % kChunks) * 8;
                return s_buf + swz((unsigned)((row * C::SW + col0 + tr) * kPB + 16 * tj));
            };
            auto dst = [&](int b) {
                const int row = b / kChunks, col0 = (b % kChunks) * 8;
                return t_slot + 2u * (unsigned)((8 * tj + tr) * C::CS + row * C::RS + col0);
            };
            for (int b = warp; b < kSteps; b += 2 * kStride) {
                unsigned v[2][4];
#pragma unroll
                for (int e = 0; e < 2; ++e) ldsm_x4_trans(v[e][0], v[e][1], v[e][2], v[e][3], src(b + e * kStride));
#pragma unroll
                for (int e = 0; e < 2; ++e) stsm_x4(dst(b + e * kStride), v[e][0], v[e][1], v[e][2], v[e][3]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfull[slot]);
            named_bar_sync(1, C::kProdThreads);  // every producer warp is done with staging slot ss
            if (tid == 0 && issued < n_pieces && !*abort) issue();
        }
        // After a wait gave up, let the copies that may still be in flight end
        // (bounded) before the CTA's shared memory goes away.
        if (tid == 0 && *abort)
            for (int j = issued >= C::NSTAGE ? issued - C::NSTAGE : 0; j < issued; ++j)
                mbar_wait(&sfull[j % C::NSTAGE], (unsigned)(j / C::NSTAGE) & 1u);
        return;
    }

    // ---------------- consumers: MMAs, output tile, TMA store ----------------
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(C::kMmaRegs));
    // The consumers form kGroups groups (warpgroups 1 and 2 apart, or one
    // group of both); a group owns kGCh of the tile's 32 channels, its part
    // of the output tile (pixels of 2 kGCh bytes, swizzled at that span), its
    // TMA store and its named barriers, so split groups drift apart and one's
    // epilogue overlaps the other's MMAs.
    constexpr int kGroups = C::kGroups, kGCh = kCh / kGroups;
    constexpr int kGThreads = (C::kThreads - C::kProdThreads) / kGroups;
    constexpr unsigned kOPB = 2 * kGCh;  // output tile pixel bytes
    const int mw = warp - C::kProdThreads / 32, mt = tid - C::kProdThreads;
    const int grp = mt / kGThreads, gt = mt % kGThreads;
    const int bar_free = 2 + 3 * grp, bar_done = 3 + 3 * grp, bar_filt = 4 + 3 * grp;
    const int gc0 = grp * kGCh, wc0 = mw * kChPerWarp;  // first channel of the group, of the warp
    const int gq = lane / 4, t4 = lane % 4;              // mma fragment coordinates
    const unsigned short *wg = static_cast<const unsigned short *>(p.w);
    unsigned short *f_s = reinterpret_cast<unsigned short *>(S + C::f_off);  // filter slab [FH FW][32]
    const unsigned f_addr = s_addr + C::f_off;
    // A operand x of a channel = one ldmatrix.x4: matrix mj (lanes 8mj..8mj+7
    // give its row addresses) holds M rows 8(mj%2)..+7 and k 8(mj/2)..+7; M
    // row i of block mj%2 is the 16-column window at column 8i of unit row
    // x + DHT (mj%2).  ldmatrix.x2 of rows x + DHT alone: matrix mj%2 = k half.
    const int mj = lane / 8, mi = lane % 8;
    const int lane_row = (mj & 1) * C::DHT;
    const unsigned lane_col = 2u * (unsigned)(8 * mi + 8 * (mj >> 1));
    const unsigned lane_col2 = 2u * (unsigned)(8 * mi + 8 * (mj & 1));
    // Output: lane (gq, t4) writes column 8gq + 2t4 + e of each row; the
    // swizzled chunk depends on neither the row nor e.
    auto oswz = [](unsigned a) {
        return kOPB == 64 ? a ^ (((a >> 7) & 3u) << 4) : a ^ (((a >> 7) & 1u) << 4);
    };
    const unsigned o_base = o_addr + (unsigned)grp * (C::o_bytes / kGroups);
    const unsigned o_lane = o_base + oswz((unsigned)(8 * gq + 2 * t4) * kOPB + 2u * (unsigned)(wc0 - gc0));
    const unsigned o_lane0 = o_lane + (gq & 1) * kOPB, o_lane1 = o_lane + (1 - (gq & 1)) * kOPB;

    Unit cur = decode(g, u_begin);
    int pc = 0, loaded_ctile = -1;
    float bias_r[kChPerWarp];
    unsigned bfr[kChPerWarp][FH][2];  // Toeplitz bands, B fragments (k 0-7, k 8-15)
    for (int u = u_begin, k = 0; u < u_end; ++u, ++k) {
        // This unit reads pieces q - 1 and q (q - 1 is new too when the unit
        // starts a column or the range).
        const bool fill = k == 0 || cur.band == 0;
        const int q = fill ? pc + 1 : pc;
        pc += fill ? 2 : 1;
        if (cur.ctile != loaded_ctile) {
            // The group's channels of every tap go to the slab with coalesced
            // loads (a warp reads 32 or 16 consecutive channels of a tap);
            // then each lane builds its B fragments from it, 4 channels of a
            // tap per 8-byte read: B[k][n] = w[fh][k - n], lane (gq, t4) holds
            // k = 2t4, 2t4+1 (+8), n = gq; for the input gradient the filter
            // is rotated by 180 degrees.  (The previous slab was read before
            // the group's last output-tile barrier.)
            loaded_ctile = cur.ctile;
            constexpr int kSlab = FH * FW * kGCh;
#pragma unroll 4
            for (int i = gt; i < kSlab; i += kGThreads) {
                const int tap = i / kGCh, c = gc0 + i % kGCh, cc = cur.ctile * kCh + c;
                f_s[tap * kCh + c] = cc < p.C ? __ldg(wg + (size_t)tap * p.C + cc) : (unsigned short)0;
            }
            named_bar_sync(bar_filt, kGThreads);
#pragma unroll
            for (int ci = 0; ci < kChPerWarp; ++ci) {
                const int cc = cur.ctile * kCh + wc0 + ci;
                bias_r[ci] = (p.bias && cc < p.C) ? p.bias[cc] : 0.f;
            }
#pragma unroll
            for (int fh = 0; fh < FH; ++fh) {
                const int sfh = p.flip ? FH - 1 - fh : fh;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    unsigned q2[2][2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int fw = 2 * t4 + e + 8 * h - gq;
                        q2[e][0] = q2[e][1] = 0u;
                        if (fw < 0 || fw >= FW) continue;
                        const int tap = sfh * FW + (p.flip ? FW - 1 - fw : fw);
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n"
                                     : "=r"(q2[e][0]), "=r"(q2[e][1])
                                     : "r"(f_addr + 2u * (unsigned)(tap * kCh + wc0)));
                    }
                    // Channel ci is half ci % 2 of word ci / 2; B pair (e = 0, 1).
                    bfr[0][fh][h] = __byte_perm(q2[0][0], q2[1][0], 0x5410);
                    bfr[1][fh][h] = __byte_perm(q2[0][0], q2[1][0], 0x7632);
                    bfr[2][fh][h] = __byte_perm(q2[0][1], q2[1][1], 0x5410);
                    bfr[3][fh][h] = __byte_perm(q2[0][1], q2[1][1], 0x7632);
                }
            }
        }
        if (fill) ring_wait(&tfull[(q - 1) % C::NSLOT], (unsigned)((q - 1) / C::NSLOT) & 1u, abort, err);
        ring_wait(&tfull[q % C::NSLOT], (unsigned)(q / C::NSLOT) & 1u, abort, err);

        // Unit row x is ring row (8 ((q - 1) % 3) + x) mod 24.
        const int rb = C::PR * ((q - 1) % C::NSLOT);
        const unsigned cb = t_addr + 2u * (unsigned)(wc0 * C::CS);
        auto op4 = [&](int ci, int x) {
            int r = rb + lane_row + x;
            r -= r >= C::TRR ? C::TRR : 0;
            return cb + lane_col + 2u * (unsigned)(ci * C::CS + r * C::RS);
        };
        auto op2 = [&](int ci, int x) {
            int r = rb + C::DHT + x;
            r -= r >= C::TRR ? C::TRR : 0;
            return cb + lane_col2 + 2u * (unsigned)(ci * C::CS + r * C::RS);
        };

        // MMAs: each step loads the next operand (also across channels) and
        // runs the MMAs of the current one; MMA (row set j, filter row fh)
        // reads operand x = j + fh.  The upper half of operand x (rows
        // x + DHT) is the lower half of operand x + DHT, so a channel's
        // operands are taken in chains x = r, r + DHT, r + 2 DHT, ...: a
        // chain's first operand is one ldmatrix.x4, every later one copies its
        // lower half from registers and loads its upper half (ldmatrix.x2).
        // The order of the MMAs on each accumulator is fixed.
        constexpr bool kChain = DWCONV_RING_CHAIN != 0;
        constexpr int NR = kChain ? (C::DHT < NQ ? C::DHT : NQ) : 1;  // chains per channel
        constexpr int XS = kChain ? C::DHT : 1;                        // operand step within a chain
        float d[kChPerWarp][C::KNB][4];
        unsigned a[4], an[4];
        ldsm_x4(a[0], a[1], a[2], a[3], op4(0, 0));
#pragma unroll
        for (int ci = 0; ci < kChPerWarp; ++ci) {
#pragma unroll
            for (int j = 0; j < C::KNB; ++j) d[ci][j][0] = d[ci][j][1] = d[ci][j][2] = d[ci][j][3] = bias_r[ci];
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int x = r; x < NQ; x += XS) {
                    bool next = true;
                    if (x + XS < NQ) {
                        if constexpr (kChain) {
                            an[0] = a[1];
                            an[2] = a[3];
                            ldsm_x2(an[1], an[3], op2(ci, x + XS));
                        } else {
                            ldsm_x4(an[0], an[1], an[2], an[3], op4(ci, x + 1));
                        }
                    } else if (r + 1 < NR) {
                        ldsm_x4(an[0], an[1], an[2], an[3], op4(ci, r + 1));
                    } else if (ci + 1 < kChPerWarp) {
                        ldsm_x4(an[0], an[1], an[2], an[3], op4(ci + 1, 0));
                    } else {
                        next = false;
                    }
#pragma unroll
                    for (int j = 0; j < C::KNB; ++j) {
                        const int fh = x - j;
                        if (fh >= 0 && fh < FH)
                            Op::run(d[ci][j], a[0], a[1], a[2], a[3], bfr[ci][fh][0], bfr[ci][fh][1]);
                    }
                    if (next)
#pragma unroll
                        for (int e = 0; e < 4; ++e) a[e] = an[e];
                }
        }
        // Piece q - 1 is not read again; piece q neither when the next unit
        // starts a column.
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&tempty[(q - 1) % C::NSLOT]);
            if (cur.band + 1 == g.tiles_h) mbar_arrive(&tempty[q % C::NSLOT]);
        }

        // Output tile, swizzled for the TMA store: this lane writes 8 bytes
        // (its warp's 4 channels) per output position, the two columns 2t4,
        // 2t4+1 in the order set by gq's parity (4-way instead of 8-way bank
        // conflicts).  Row set j is output rows j and j + 4.
        if (gt == 0) asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
        named_bar_sync(bar_free, kGThreads);  // the previous unit's store has read the tile
#pragma unroll
        for (int j = 0; j < C::KNB; ++j)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                unsigned lo[2], hi[2];  // column 2t4 + e: channels (0, 1), (2, 3)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    lo[e] = Op::pack(d[0][j][2 * half + e], d[1][j][2 * half + e]);
                    hi[e] = Op::pack(d[2][j][2 * half + e], d[3][j][2 * half + e]);
                }
                const bool odd = gq & 1;
                const unsigned row = (unsigned)((j + half * C::DHT) * C::OTW) * kOPB;
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};\n" ::"r"(o_lane0 + row), "r"(odd ? lo[1] : lo[0]),
                             "r"(odd ? hi[1] : hi[0])
                             : "memory");
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};\n" ::"r"(o_lane1 + row), "r"(odd ? lo[0] : lo[1]),
                             "r"(odd ? hi[0] : hi[1])
                             : "memory");
            }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // visible to the TMA store
        named_bar_sync(bar_done, kGThreads);                             // output tile complete
        if (gt == 0) {
            asm volatile(
                "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];\n" ::"l"(
                    reinterpret_cast<uint64_t>(&out_map)),
                "r"(cur.ctile * kCh + gc0), "r"(cur.twi * C::OTW), "r"(cur.band * C::PR), "r"(cur.group),
                "r"(o_base)
                : "memory");
            asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
        }
        advance(g, g.groups, cur);
    }
    if (gt == 0) asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}

// Registers per thread the kernel is compiled to launch with (read once).
template <typename K>
int launch_regs(K kern) {
    static std::atomic<int> regs{-1};
    int r = regs.load(std::memory_order_relaxed);
    if (r < 0) {
        cudaFuncAttributes a{};
        if (cudaFuncGetAttributes(&a, reinterpret_cast<const void *>(kern)) != cudaSuccess) return 0;
        r = a.numRegs;
        regs.store(r, std::memory_order_relaxed);
    }
    return r;
}

template <typename T, int FH, int FW>
cudaError_t run_ring(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    using C = CfgR;
    GeoM g{};
    g.tiles_h = (p.OHs + C::PR - 1) / C::PR;
    g.tiles_w = (p.OWs + C::OTW - 1) / C::OTW;
    g.groups = p.N;
    const long long per = (long long)g.groups * g.tiles_w * g.tiles_h;
    const long long units = per * ((p.C + kCh - 1) / kCh);
    if (units >= (1LL << 30)) return cudaErrorNotSupported;
    g.per_ctile = (int)per;
    g.units = (int)units;
    const uint32_t box[4] = {(uint32_t)kCh, (uint32_t)C::SW, (uint32_t)C::PR, 1u};
    constexpr int kGCh = kCh / C::kGroups;  // channels of one consumer group's output tile
    const uint32_t obox[4] = {(uint32_t)kGCh, (uint32_t)C::OTW, (uint32_t)C::PR, 1u};
    CUtensorMap map, omap;
    if (!make_mma_halo_map(&map, p, dt, sizeof(T), box, kPB) ||
        !make_out_map(&omap, p, dt, sizeof(T), obox, 2 * kGCh))
        return cudaErrorNotSupported;
    auto kern = tiled_mma_ring_kernel<T, FH, FW>;
    // setmaxnreg redistributes the registers the CTA was launched with: the
    // split is only valid for the register count it was sized against.
    if (launch_regs(kern) != C::kLaunchRegs) return cudaErrorNotSupported;
    int per_sm = 0;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), C::kThreads, C::smem + 1024, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const int grid = (int)std::min<long long>(g.units, (long long)sm_count() * per_sm);
    kern<<<grid, C::kThreads, C::smem + 1024, st>>>(map, omap, p, g, device_error_word());
    note_launches(1);
    note_kernel("tiled_mma_ring");
    return cudaGetLastError();
}

// Plain (unfused) 16-bit passes: the warp-specialised ring kernel for 5x5 and
// 7x7 filters on maps wider than 32 columns, tiled_mma_kernel otherwise (or if
// the ring kernel's register split is not available).  Measured on GB300
// (x[128,56,56,96]): 7x7 forward 45.3 against 47.1 us, input gradient 45.1
// against 48.7 us; 5x5 forward 38.9 against 40.9 us; 3x3 forward 37.2 against
// 34.4 us (too few MMAs per unit to cover the pipeline), so 3x3 stays on
// tiled_mma_kernel.
template <typename T>
cudaError_t by_filter_plain(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (DWCONV_MMA_RING && p.OWs > 32) {
        cudaError_t e = cudaErrorNotSupported;
        if (p.FH == 7 && p.FW == 7)
            e = run_ring<T, 7, 7>(p, dt, st);
        else if (p.FH == 5 && p.FW == 5)
            e = run_ring<T, 5, 5>(p, dt, st);
        if (e != cudaErrorNotSupported) return e;
    }
    return by_filter<T, false>(p, dt, st);
}

}  // namespace
}  // namespace dwc
