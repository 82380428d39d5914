// Stride-2, dilation-1 passes of 3x3, 5x5 and 7x7 filters: forward, input
// gradient and weight gradient, register-tiled on the CUDA cores.
//
// These layers are HBM-bound (a few multiply-adds per byte), so what matters is
// that every tensor is read or written once, with whole-sector accesses: each
// unit's input block is staged in shared memory by one TMA tensor copy (zero
// fill outside the tensor = generated padding), double-buffered, with bounded
// waits, as in the unit-stride kernels (tiled_common.cuh).
//
// Forward.  An output tile of T rows reads (T - 1) S + F input rows
// ("Tiles, halos and partial sums": the halo of a stride-2 2x2 tile of a 3x3
// filter spans 5x5 inputs).  A thread owns a channel pair and TH x TW outputs;
// it walks its (TH - 1) 2 + F input rows once, each row's (TW - 1) 2 + F values
// read from shared memory once and fed to every (output row, filter row) pair
// that uses them -- the row-stationary reuse of the unit-stride kernels with
// every other input column.
//
// Input gradient.  dx at input row 2a + phi receives taps fh = rho + 2u (rho =
// (phi + P) mod 2) from dy row a + floor((phi + P)/2) - u, so each of the four
// output phases (phi_h, phi_w) of dx is a unit-stride correlation of dy with a
// sub-filter of the taps of one parity (Flash-DWC §5.1 reads the input
// gradient as a convolution of dy with the rotated filter; with stride 2 it
// splits into these four).  A CTA's 8 thread tiles are the 4 phases x 2 tiles,
// all reading one staged dy block, so dx is written exactly once and dy read
// once; a phase whose sub-filter is smaller than the largest one computes with
// zero taps (2 x 2 sub-filters for 3x3: 16 products for 9 taps per 2x2 dx block).
//
// Weight gradient.  dw[fh,fw,c] = sum over (n, i, j) of dy[n,i,j,c] *
// x[n, 2i - P + fh, 2j - P + fw, c]: the forward pass's tiling with the roles
// of filter and output exchanged, as in tiled_wgrad.cu -- per-thread fp32
// accumulators for all F x F taps, the N*OH*OW axis split into Zc slices
// (Flash-DWC §5.1), a fixed-order reduction inside the CTA and then across the
// slices (wgrad_reduce), so results are bit-identical from call to call.
//
// Every multiply-add accumulates in fp32 (Mac<T> in common.cuh); the forward
// pass adds the bias once, at the start.
#include "tiled_common.cuh"

namespace dwc {
namespace {

using namespace tiled;

constexpr int kS = 2;  // stride

// Geometry of a unit grid: NI * RT * CT thread tiles of TH x TW outputs (of
// the output, or of one phase of dx), HH x HW staged rows / columns per image.
// `rows_for(tile_rows)` / `cols_for(tile_cols)` give the staged extent of a
// unit of that many output rows / columns.  Thread tiles are arranged columns
// first, then rows, then images (as make_geo), within `tiles` tiles and the
// double-buffered stage within `smem_cap` bytes.
template <typename RowsFor, typename ColsFor>
Geo make_geo_s(int N, int OHs, int OWs, int C, int TH, int TW, int tiles, size_t elem, size_t extra_px,
               size_t smem_cap, RowsFor rows_for, ColsFor cols_for) {
    Geo g{};
    auto arrange = [&](int CT) {
        g.CT = CT;
        g.RT = std::min(tiles / g.CT, next_pow2((OHs + TH - 1) / TH));
        g.NI = tiles / (g.CT * g.RT);
        g.HH = rows_for(g.RT * TH);
        g.HW = cols_for(g.CT * TW);
    };
    auto stage = [&]() {
        const size_t px = (size_t)g.HH * g.HW + extra_px * (size_t)(g.RT * TH) * (g.CT * TW);
        return 2 * (size_t)g.NI * px * 32 * elem;
    };
    arrange(std::min(tiles, next_pow2((OWs + TW - 1) / TW)));
    while (stage() > smem_cap && g.CT > 1) arrange(g.CT / 2);
    g.tiles_h = (OHs + g.RT * TH - 1) / (g.RT * TH);
    g.tiles_w = (OWs + g.CT * TW - 1) / (g.CT * TW);
    g.groups = (N + g.NI - 1) / g.NI;
    g.ctiles = (C + 31) / 32;
    const long long per = (long long)g.groups * g.tiles_w * g.tiles_h;
    const long long units = per * g.ctiles;
    g.per_ctile = (int)std::min<long long>(per, 1LL << 30);
    g.units = units < (1LL << 30) ? (int)units : 0;
    return g;
}

// Tensor map of an NHWC tensor [N][H][W][C]; one box = [NI][rows][cols][32];
// `promo`: L2 promotion of the copies in bytes.
bool make_nhwc_map(CUtensorMap *m, const void *base, int N, int H, int W, int C, int rows, int cols, int NI,
                   dwconv_dtype dt, size_t es, int promo = DWCONV_L2_PROMO) {
    const uint64_t dims[4] = {(uint64_t)C, (uint64_t)W, (uint64_t)H, (uint64_t)N};
    const uint64_t str[3] = {(uint64_t)C * es, (uint64_t)W * C * es, (uint64_t)H * W * C * es};
    const uint32_t box[4] = {32, (uint32_t)cols, (uint32_t)rows, (uint32_t)NI};
    return encode_tmap_4d(m, dt, base, dims, str, box, 0, promo);
}

// Arguments of one strided pass (sizes as in Shape; pad per axis).
struct SArgs {
    const void *in;     // x (forward, weight gradient) or dy (input gradient)
    const void *w;      // filter (forward, input gradient)
    const void *dy;     // weight gradient: dy
    const float *bias;  // forward, nullable
    Fuse fz;            // forward: BN+Act prologue, affine+activation epilogue
    void *out;          // y, dx
    int N, H, W, C, OH, OW, PH, PW;
};

// ---------------------------------------------------------------- forward

// FUSE: the fused forward pass (Flash-DWC §5.2) -- the BN+Act prologue on the
// staged halo (in place, padding kept zero) and the affine+activation
// epilogue on the fp32 sums; 1: piecewise-linear activations only, 2: all;
// 0: plain (separate instances, so the plain pass keeps its code).
template <typename T, int F, int TH, int TW, int MINB, int FUSE>
__global__ void __launch_bounds__(kThreads, MINB)
    strided_fwd_kernel(const __grid_constant__ CUtensorMap halo_map, SArgs a, Geo g, unsigned *err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2];
    constexpr int WR = (TH - 1) * kS + F, WW = (TW - 1) * kS + F;  // thread's input window

    const int tid = threadIdx.x, cp = tid % kPairs, t = tid / kPairs;
    const int img_l = t / (g.RT * g.CT), rt = (t / g.CT) % g.RT, ct = t % g.CT;
    const int tile_rows = g.RT * TH, tile_cols = g.CT * TW;
    const unsigned box_bytes = halo_box_bytes(g, sizeof(T));
    const unsigned buf_stride = align128(box_bytes);
    const int halo_elems = g.HH * g.HW * 32;
    const T *wgt = static_cast<const T *>(a.w);
    T *out = static_cast<T *>(a.out);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    auto issue = [&](int u, int b) {
        const Unit un = decode(g, u);
        mbar_arrive_expect_tx(&bars[b], box_bytes);
        tma_load_4d(smem_raw + b * buf_stride, &halo_map, un.ctile * 32, un.twi * tile_cols * kS - a.PW,
                    un.band * tile_rows * kS - a.PH, un.group * g.NI, &bars[b]);
    };

    using M = Mac<T>;
    typename M::V wr[F][F];
    float2 bias2 = make_float2(0.f, 0.f);
    int loaded_ctile = -1;

    const int u_end = (int)((long long)g.units * (blockIdx.x + 1) / gridDim.x);
    int u = (int)((long long)g.units * blockIdx.x / gridDim.x);
    if (tid == 0 && u < u_end) issue(u, 0);
    for (int k = 0; u < u_end; ++k, ++u) {
        const int un = u + 1 < u_end ? u + 1 : g.units;
        if (tid == 0 && un < g.units) issue(un, (k + 1) & 1);
        if (!mbar_wait(&bars[k & 1], (k >> 1) & 1)) {
            report_timeout(err);
            if (tid == 0 && un < g.units) mbar_wait(&bars[(k + 1) & 1], ((k + 1) >> 1) & 1);
            return;
        }
        const Unit cur = decode(g, u);
        const int c = cur.ctile * 32 + 2 * cp;
        const bool cvalid = c < a.C;
        if constexpr (FUSE > 0) {
            if (a.fz.pre()) {
                // BN+Act prologue once per staged value, in place: thread (cp, t)
                // takes channel pair cp of every kTiles-th halo row.  Positions
                // outside the input are padding of x' and stay zero; x' is
                // rounded to T as the unfused layer would store it.
                T *hbuf = reinterpret_cast<T *>(smem_raw + (k & 1) * buf_stride);
                const Affine a0 = cvalid ? affine_in(a.fz, c) : Affine{1.f, 0.f};
                const Affine a1 = cvalid ? affine_in(a.fz, c + 1) : Affine{1.f, 0.f};
                const float2 s2 = make_float2(a0.s, a1.s), t2 = make_float2(a0.t, a1.t);
                // Halo columns [c_lo, c_hi) lie inside the input.
                const int col_in = cur.twi * tile_cols * kS - a.PW;
                const int c_lo = min(max(-col_in, 0), g.HW), c_hi = max(min(a.W - col_in, g.HW), c_lo);
                with_act<FUSE == 1>(a.fz.in_act, [&](auto act) {
                    [[maybe_unused]] constexpr int A = decltype(act)::value;
#pragma unroll 1
                    for (int rr = t; rr < g.NI * g.HH; rr += kTiles) {
                        const int im = rr / g.HH, r = rr - im * g.HH;
                        const int ih = cur.band * tile_rows * kS - a.PH + r;
                        const bool rok = ih >= 0 && ih < a.H && cur.group * g.NI + im < a.N;
                        T *row = hbuf + rr * g.HW * 32 + 2 * cp;
                        const int lo = rok ? c_lo : g.HW, hi = rok ? c_hi : g.HW;
#pragma unroll 1
                        for (int col = 0; col < lo; ++col) Pair<T>::store(row + col * 32, make_float2(0.f, 0.f));
#pragma unroll 4
                        for (int col = lo; col < hi; ++col) {
                            if constexpr (sizeof(T) == 4) {
                                float2 *q = reinterpret_cast<float2 *>(row + col * 32);
                                *q = prologue_f32<A>(*q, s2, t2);
                            } else {
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
        }
        if (cur.ctile != loaded_ctile) {
            loaded_ctile = cur.ctile;
#pragma unroll
            for (int fh = 0; fh < F; ++fh)
#pragma unroll
                for (int fw = 0; fw < F; ++fw) wr[fh][fw] = cvalid ? M::load(wgt + (fh * F + fw) * a.C + c) : M::zero();
            bias2 = (a.bias && cvalid) ? make_float2(a.bias[c], a.bias[c + 1]) : make_float2(0.f, 0.f);
        }
        const T *s = reinterpret_cast<const T *>(smem_raw + (k & 1) * buf_stride) + img_l * halo_elems;
        const int r0 = rt * TH * kS, j0 = ct * TW * kS;
        float2 acc[TH][TW];
#pragma unroll
        for (int th = 0; th < TH; ++th)
#pragma unroll
            for (int tw = 0; tw < TW; ++tw) acc[th][tw] = bias2;
#pragma unroll
        for (int r = 0; r < WR; ++r) {
            typename M::V xv[WW];
            const T *srow = s + ((r0 + r) * g.HW + j0) * 32 + 2 * cp;
#pragma unroll
            for (int j = 0; j < WW; ++j) xv[j] = M::load(srow + j * 32);
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int fh = r - kS * th;
                if (fh < 0 || fh >= F) continue;
#pragma unroll
                for (int fw = 0; fw < F; ++fw)
#pragma unroll
                    for (int tw = 0; tw < TW; ++tw) M::fma(acc[th][tw], wr[fh][fw], xv[kS * tw + fw]);
            }
        }
        const int n = cur.group * g.NI + img_l;
        if (cvalid && n < a.N) {
            if (FUSE > 0 && a.fz.post()) {
                const Affine o0 = affine_out(a.fz, c), o1 = affine_out(a.fz, c + 1);
                with_act<FUSE == 1>(a.fz.out_act, [&](auto act) {
                    constexpr int A = decltype(act)::value;
#pragma unroll
                    for (int th = 0; th < TH; ++th)
#pragma unroll
                        for (int tw = 0; tw < TW; ++tw) {
                            acc[th][tw].x = activate(fmaf(o0.s, acc[th][tw].x, o0.t), A);
                            acc[th][tw].y = activate(fmaf(o1.s, acc[th][tw].y, o1.t), A);
                        }
                });
            }
            const int i0 = cur.band * tile_rows + rt * TH, jj0 = cur.twi * tile_cols + ct * TW;
            T *img = out + (long long)n * a.OH * a.OW * a.C + c;
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int i = i0 + th;
                if (i >= a.OH) break;
#pragma unroll
                for (int tw = 0; tw < TW; ++tw) {
                    const int j = jj0 + tw;
                    if (j >= a.OW) break;
                    Pair<T>::store(img + ((long long)i * a.OW + j) * a.C, acc[th][tw]);
                }
            }
        }
        __syncthreads();  // this buffer is refilled by the copy issued next iteration
    }
}

// ---------------------------------------------------------- input gradient

// Thread tile t = tid / 16 of a CTA: phase (phi_h, phi_w) = ((t >> 1) & 1, t & 1)
// and spatial tile t >> 2 (of NI * RT * CT = 2).  Positions are counted on the
// phase grid: phase position (a, b) is dx[2a + phi_h][2b + phi_w].  With
// kh(phi) = floor((phi + P) / 2) and NU = ceil(F / 2), the sub-filter of phase
// phi_h holds the taps fh = rho + 2u (rho = (phi_h + P) mod 2, u < NU, zero
// where fh >= F), and dx at phase row a takes dy rows a + kh(phi_h) - u.  A
// unit of TA phase rows starting at A0 reads dy rows from A0 + floor(P/2) -
// NU + 1 on: TA + (P mod 2) + NU - 1 of them (columns alike).
template <typename T, int F, int TH, int TW, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    strided_dgrad_kernel(const __grid_constant__ CUtensorMap dy_map, SArgs a, Geo g, unsigned *err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2];
    constexpr int NU = (F + 1) / 2;
    constexpr int WR = TH + NU - 1, WW = TW + NU - 1;  // thread's dy window

    const int tid = threadIdx.x, cp = tid % kPairs, t = tid / kPairs;
    const int phi_h = (t >> 1) & 1, phi_w = t & 1, q = t >> 2;
    const int img_l = q / (g.RT * g.CT), rt = (q / g.CT) % g.RT, ct = q % g.CT;
    const int tile_rows = g.RT * TH, tile_cols = g.CT * TW;  // phase positions per unit
    const int rho_h = (phi_h + a.PH) & 1, rho_w = (phi_w + a.PW) & 1;
    // Offset of this phase's window in the staged block: kh(phi) - floor(P/2).
    const int dh = ((phi_h + a.PH) >> 1) - (a.PH >> 1), dw = ((phi_w + a.PW) >> 1) - (a.PW >> 1);
    const unsigned box_bytes = halo_box_bytes(g, sizeof(T));
    const unsigned buf_stride = align128(box_bytes);
    const int halo_elems = g.HH * g.HW * 32;
    const T *wgt = static_cast<const T *>(a.w);
    T *out = static_cast<T *>(a.out);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    auto issue = [&](int u, int b) {
        const Unit un = decode(g, u);
        mbar_arrive_expect_tx(&bars[b], box_bytes);
        tma_load_4d(smem_raw + b * buf_stride, &dy_map, un.ctile * 32,
                    un.twi * tile_cols + (a.PW >> 1) - NU + 1, un.band * tile_rows + (a.PH >> 1) - NU + 1,
                    un.group * g.NI, &bars[b]);
    };

    using M = Mac<T>;
    typename M::V wr[NU][NU];  // this phase's sub-filter, zero where the tap does not exist
    int loaded_ctile = -1;

    const int u_end = (int)((long long)g.units * (blockIdx.x + 1) / gridDim.x);
    int u = (int)((long long)g.units * blockIdx.x / gridDim.x);
    if (tid == 0 && u < u_end) issue(u, 0);
    for (int k = 0; u < u_end; ++k, ++u) {
        const int un = u + 1 < u_end ? u + 1 : g.units;
        if (tid == 0 && un < g.units) issue(un, (k + 1) & 1);
        if (!mbar_wait(&bars[k & 1], (k >> 1) & 1)) {
            report_timeout(err);
            if (tid == 0 && un < g.units) mbar_wait(&bars[(k + 1) & 1], ((k + 1) >> 1) & 1);
            return;
        }
        const Unit cur = decode(g, u);
        const int c = cur.ctile * 32 + 2 * cp;
        const bool cvalid = c < a.C;
        if (cur.ctile != loaded_ctile) {
            loaded_ctile = cur.ctile;
#pragma unroll
            for (int uu = 0; uu < NU; ++uu)
#pragma unroll
                for (int vv = 0; vv < NU; ++vv) {
                    const int fh = rho_h + 2 * uu, fw = rho_w + 2 * vv;
                    wr[uu][vv] = (cvalid && fh < F && fw < F) ? M::load(wgt + (fh * F + fw) * a.C + c) : M::zero();
                }
        }
        const T *s = reinterpret_cast<const T *>(smem_raw + (k & 1) * buf_stride) + img_l * halo_elems;
        const int r0 = rt * TH + dh, j0 = ct * TW + dw;
        float2 acc[TH][TW];
#pragma unroll
        for (int th = 0; th < TH; ++th)
#pragma unroll
            for (int tw = 0; tw < TW; ++tw) acc[th][tw] = make_float2(0.f, 0.f);
        // dx at (th, tw) takes tap (u, v) from window position (th + NU-1 - u, tw + NU-1 - v).
#pragma unroll
        for (int r = 0; r < WR; ++r) {
            typename M::V xv[WW];
            const T *srow = s + ((r0 + r) * g.HW + j0) * 32 + 2 * cp;
#pragma unroll
            for (int j = 0; j < WW; ++j) xv[j] = M::load(srow + j * 32);
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int uu = th + NU - 1 - r;
                if (uu < 0 || uu >= NU) continue;
#pragma unroll
                for (int vv = 0; vv < NU; ++vv)
#pragma unroll
                    for (int tw = 0; tw < TW; ++tw) M::fma(acc[th][tw], wr[uu][vv], xv[tw + NU - 1 - vv]);
            }
        }
        const int n = cur.group * g.NI + img_l;
        if (cvalid && n < a.N) {
            const int pa0 = cur.band * tile_rows + rt * TH, pb0 = cur.twi * tile_cols + ct * TW;
            T *img = out + (long long)n * a.H * a.W * a.C + c;
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int i = 2 * (pa0 + th) + phi_h;
                if (i >= a.H) break;
#pragma unroll
                for (int tw = 0; tw < TW; ++tw) {
                    const int j = 2 * (pb0 + tw) + phi_w;
                    if (j >= a.W) break;
                    Pair<T>::store(img + ((long long)i * a.W + j) * a.C, acc[th][tw]);
                }
            }
        }
        __syncthreads();  // this buffer is refilled by the copy issued next iteration
    }
}

// --------------------------------------------------------- weight gradient

template <typename T, int F, int TH, int TW, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    strided_wgrad_kernel(const __grid_constant__ CUtensorMap halo_map, const __grid_constant__ CUtensorMap dy_map,
                         SArgs a, Geo g, float *__restrict__ part, int Zc, unsigned *err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2];
    constexpr int WR = (TH - 1) * kS + F, WW = (TW - 1) * kS + F;

    const int tid = threadIdx.x, cp = tid % kPairs, t = tid / kPairs;
    const int img_l = t / (g.RT * g.CT), rt = (t / g.CT) % g.RT, ct = t % g.CT;
    const int tile_rows = g.RT * TH, tile_cols = g.CT * TW;
    const int halo_elems = g.HH * g.HW * 32, otile_elems = tile_rows * tile_cols * 32;
    const unsigned hb = halo_box_bytes(g, sizeof(T)), tb = tile_box_bytes(g, TH, TW, sizeof(T));
    const unsigned stage = align128(hb) + align128(tb);
    const int ctile = blockIdx.x / Zc, z = blockIdx.x % Zc;
    const int base = ctile * g.per_ctile;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    auto issue = [&](int v, int b) {
        const Unit un = decode(g, base + v);
        mbar_arrive_expect_tx(&bars[b], hb + tb);
        unsigned char *dst = smem_raw + b * stage;
        tma_load_4d(dst, &halo_map, un.ctile * 32, un.twi * tile_cols * kS - a.PW, un.band * tile_rows * kS - a.PH,
                    un.group * g.NI, &bars[b]);
        tma_load_4d(dst + align128(hb), &dy_map, un.ctile * 32, un.twi * tile_cols, un.band * tile_rows,
                    un.group * g.NI, &bars[b]);
    };

    using M = Mac<T>;
    float2 acc[F][F];
#pragma unroll
    for (int fh = 0; fh < F; ++fh)
#pragma unroll
        for (int fw = 0; fw < F; ++fw) acc[fh][fw] = make_float2(0.f, 0.f);

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
        const int i0 = rt * TH, j0 = ct * TW;
        typename M::V dyv[TH][TW];
#pragma unroll
        for (int th = 0; th < TH; ++th)
#pragma unroll
            for (int tw = 0; tw < TW; ++tw) dyv[th][tw] = M::load(sy + ((i0 + th) * tile_cols + j0 + tw) * 32 + 2 * cp);
#pragma unroll
        for (int r = 0; r < WR; ++r) {
            typename M::V xv[WW];
            const T *srow = sx + ((i0 * kS + r) * g.HW + j0 * kS) * 32 + 2 * cp;
#pragma unroll
            for (int j = 0; j < WW; ++j) xv[j] = M::load(srow + j * 32);
#pragma unroll
            for (int th = 0; th < TH; ++th) {
                const int fh = r - kS * th;
                if (fh < 0 || fh >= F) continue;
#pragma unroll
                for (int fw = 0; fw < F; ++fw)
#pragma unroll
                    for (int tw = 0; tw < TW; ++tw) M::fma(acc[fh][fw], dyv[th][tw], xv[kS * tw + fw]);
            }
        }
        __syncthreads();  // this buffer is refilled by the copy issued next iteration
    }

    // Sum the 8 thread tiles of each channel pair: lanes l and l^16 of a warp
    // hold tiles 2w and 2w+1; then the four warps, in a fixed order.
    float2 *red = reinterpret_cast<float2 *>(smem_raw);  // [4][F*F][16]
    const int warp = tid / 32, lane = tid % 32;
#pragma unroll
    for (int fh = 0; fh < F; ++fh)
#pragma unroll
        for (int fw = 0; fw < F; ++fw) {
            float2 s = acc[fh][fw];
            s.x += __shfl_xor_sync(0xffffffffu, s.x, 16);
            s.y += __shfl_xor_sync(0xffffffffu, s.y, 16);
            if (lane < 16) red[(warp * F * F + fh * F + fw) * 16 + lane] = s;
        }
    __syncthreads();
    for (int idx = tid; idx < F * F * 16; idx += kThreads) {
        const int tap = idx / 16, pr = idx % 16;
        float2 s = red[tap * 16 + pr];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) {
            const float2 o = red[(w * F * F + tap) * 16 + pr];
            s.x += o.x;
            s.y += o.y;
        }
        const int c = ctile * 32 + 2 * pr;
        if (c < a.C) {
            float *dst = part + ((long long)z * F * F + tap) * a.C + c;
            dst[0] = s.x;
            dst[1] = s.y;
        }
    }
}

// ---------------------------------------------------------------- launchers

// Thread tiles and CTAs per SM (register budget): 16-bit data keeps pairs
// packed in 32-bit registers, fp32 data in float2.
#ifndef DWCONV_ST_CAP_KB
#define DWCONV_ST_CAP_KB 72  // cap on a CTA's two stages
#endif
#ifndef DWCONV_ST_FWD_TH16
#define DWCONV_ST_FWD_TH16 2
#endif
#ifndef DWCONV_ST_DG_TH
#define DWCONV_ST_DG_TH 4
#endif
template <typename T> constexpr bool packed() { return sizeof(T) == 2; }
template <typename T> constexpr int fwd_th() { return packed<T>() ? DWCONV_ST_FWD_TH16 : 1; }
constexpr int kTW = 7;

template <typename T>
size_t stage_cap() {
    return DWCONV_ST_CAP_KB * 1024;
}

int rows_halo(int tile, int F) { return (tile - 1) * kS + F; }

template <typename T, int F, int TH, int TW, int MINB, int FUSE>
cudaError_t run_fwd(const SArgs &a, dwconv_dtype dt, cudaStream_t st) {
    const Geo g = make_geo_s(a.N, a.OH, a.OW, a.C, TH, TW, kTiles, sizeof(T), 0, stage_cap<T>(),
                             [](int r) { return rows_halo(r, F); }, [](int c) { return rows_halo(c, F); });
    if (g.units == 0) return cudaErrorNotSupported;
    const size_t smem = 2 * (size_t)align128(halo_box_bytes(g, sizeof(T)));
    if (smem > 220 * 1024 || g.HH > 256 || g.HW > 256) return cudaErrorNotSupported;
    CUtensorMap map;
    if (!make_nhwc_map(&map, a.in, a.N, a.H, a.W, a.C, g.HH, g.HW, g.NI, dt, sizeof(T))) return cudaErrorNotSupported;
    auto kern = strided_fwd_kernel<T, F, TH, TW, MINB, FUSE>;
    int per_sm = 0;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kThreads, smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const int grid = (int)std::min<long long>(g.units, (long long)sm_count() * per_sm);
    kern<<<grid, kThreads, smem, st>>>(map, a, g, device_error_word());
    note_launches(1);
    note_kernel("strided_fwd");
    return cudaGetLastError();
}

template <typename T, int F, int TH, int TW, int MINB>
cudaError_t run_dgrad(const SArgs &a, dwconv_dtype dt, cudaStream_t st) {
    constexpr int NU = (F + 1) / 2;
    const int ph = a.PH & 1, pw = a.PW & 1;
    const Geo g = make_geo_s(a.N, (a.H + 1) / 2, (a.W + 1) / 2, a.C, TH, TW, 2, sizeof(T), 0, stage_cap<T>(),
                             [&](int r) { return r + ph + NU - 1; }, [&](int c) { return c + pw + NU - 1; });
    if (g.units == 0) return cudaErrorNotSupported;
    const size_t smem = 2 * (size_t)align128(halo_box_bytes(g, sizeof(T)));
    if (smem > 220 * 1024 || g.HH > 256 || g.HW > 256) return cudaErrorNotSupported;
    CUtensorMap map;
    if (!make_nhwc_map(&map, a.in, a.N, a.OH, a.OW, a.C, g.HH, g.HW, g.NI, dt, sizeof(T)))
        return cudaErrorNotSupported;
    auto kern = strided_dgrad_kernel<T, F, TH, TW, MINB>;
    int per_sm = 0;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kThreads, smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const int grid = (int)std::min<long long>(g.units, (long long)sm_count() * per_sm);
    kern<<<grid, kThreads, smem, st>>>(map, a, g, device_error_word());
    note_launches(1);
    note_kernel("strided_dgrad");
    return cudaGetLastError();
}

// Weight-gradient plan: geometry and the slice count Zc (about one wave of the
// CTAs that fit on the SMs, over all channel tiles), for the workspace bound or
// the current device (plan_sms).
template <typename T, int F, int TH, int TW, int MINB>
bool plan_wgrad(const SArgs &a, Geo &g, int &Zc, size_t &smem, bool launch) {
    g = make_geo_s(a.N, a.OH, a.OW, a.C, TH, TW, kTiles, sizeof(T), 1, stage_cap<T>(),
                   [](int r) { return rows_halo(r, F); }, [](int c) { return rows_halo(c, F); });
    if (g.units == 0 || g.HH > 256 || g.HW > 256) return false;
    smem = 2 * (size_t)(align128(halo_box_bytes(g, sizeof(T))) + align128(tile_box_bytes(g, TH, TW, sizeof(T))));
    smem = std::max(smem, (size_t)(kThreads / 32) * F * F * 16 * sizeof(float2));
    if (smem > 220 * 1024) return false;
    const int resident = std::max(1, std::min(MINB, (int)(plan_smem_per_sm(launch) / (smem + 1024))));
    long long zc = (long long)plan_sms(launch) * resident / g.ctiles;
    Zc = (int)std::max(1LL, std::min<long long>(zc, g.per_ctile));
    return true;
}

template <typename T, int F, int TH, int TW, int MINB>
cudaError_t run_wgrad(const SArgs &a, dwconv_dtype dt, float *part, float *dw, cudaStream_t st) {
    Geo g;
    int Zc;
    size_t smem;
    if (!plan_wgrad<T, F, TH, TW, MINB>(a, g, Zc, smem, true)) return cudaErrorNotSupported;
    CUtensorMap halo_map, dy_map;
    // 128-byte L2 promotion for x: measured on GB300, bf16 3x3 on x[128,56,56,96],
    // 29.5 against 32.8 us with 64 bytes (the forward passes do not gain from it).
    if (!make_nhwc_map(&halo_map, a.in, a.N, a.H, a.W, a.C, g.HH, g.HW, g.NI, dt, sizeof(T), 128) ||
        !make_nhwc_map(&dy_map, a.dy, a.N, a.OH, a.OW, a.C, g.RT * TH, g.CT * TW, g.NI, dt, sizeof(T)))
        return cudaErrorNotSupported;
    auto kern = strided_wgrad_kernel<T, F, TH, TW, MINB>;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kThreads, smem, nullptr);
    if (e != cudaSuccess) return e;
    kern<<<g.ctiles * Zc, kThreads, smem, st>>>(halo_map, dy_map, a, g, part, Zc, device_error_word());
    note_launches(1);
    note_kernel("strided_wgrad");
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_wgrad_reduce(part, Zc, (long long)F * F * a.C, dw, st);
}

// Instances: 3x3, 5x5, 7x7; CTAs per SM sized to the registers each needs.
template <typename T, typename Fn>
cudaError_t by_filter(int F, Fn &&fn) {
    switch (F) {
        case 3: return fn(std::integral_constant<int, 3>{});
        case 5: return fn(std::integral_constant<int, 5>{});
        case 7: return fn(std::integral_constant<int, 7>{});
        default: return cudaErrorNotSupported;
    }
}

template <typename Fn>
cudaError_t by_dtype(dwconv_dtype dt, Fn &&fn) {
    switch (dt) {
        case DWCONV_FP32: return fn(float{});
        case DWCONV_FP16: return fn(__half{});
        case DWCONV_BF16: return fn(__nv_bfloat16{});
        default: return cudaErrorNotSupported;
    }
}

template <typename T, int F> constexpr int fwd_minb() { return packed<T>() || F < 7 ? 4 : 3; }
template <typename T, int F> constexpr int wgrad_th() { return packed<T>() ? 2 : 1; }
template <typename T, int F> constexpr int wgrad_minb() { return F < 7 ? 4 : 3; }
constexpr int kDgTH = DWCONV_ST_DG_TH, kDgMinb = 4;

bool covered(const Shape &s, dwconv_dtype dt) {
    return s.SH == kS && s.SW == kS && s.DH == 1 && s.DW == 1 && s.FH == s.FW &&
           (s.FH == 3 || s.FH == 5 || s.FH == 7) && (dt == DWCONV_FP32 || dt == DWCONV_FP16 || dt == DWCONV_BF16);
}

SArgs args_of(const Shape &s) {
    SArgs a{};
    a.N = s.N; a.H = s.H; a.W = s.W; a.C = s.C; a.OH = s.OH; a.OW = s.OW; a.PH = s.PH; a.PW = s.PW;
    return a;
}

}  // namespace

cudaError_t launch_strided_fwd(const Shape &s, dwconv_dtype dt, const void *x, const void *w, const float *bias,
                               void *y, const Fuse &fz, cudaStream_t st) {
    if (!covered(s, dt)) return cudaErrorNotSupported;
    SArgs a = args_of(s);
    a.in = x; a.w = w; a.bias = bias; a.out = y; a.fz = fz;
    const int epi = !fz.pre() && !fz.post() ? 0 : act_is_light(fz.in_act) && act_is_light(fz.out_act) ? 1 : 2;
    return by_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        return by_filter<T>(s.FH, [&](auto f) {
            constexpr int F = decltype(f)::value;
            constexpr int TH = fwd_th<T>(), MB = fwd_minb<T, F>();
            if (epi == 0) return run_fwd<T, F, TH, kTW, MB, 0>(a, dt, st);
            if (epi == 1) return run_fwd<T, F, TH, kTW, MB, 1>(a, dt, st);
            return run_fwd<T, F, TH, kTW, MB, 2>(a, dt, st);
        });
    });
}

cudaError_t launch_strided_dgrad(const Shape &s, dwconv_dtype dt, const void *dy, const void *w, void *dx,
                                 cudaStream_t st) {
    if (!covered(s, dt)) return cudaErrorNotSupported;
    SArgs a = args_of(s);
    a.in = dy; a.w = w; a.out = dx;
    return by_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        return by_filter<T>(s.FH, [&](auto f) {
            constexpr int F = decltype(f)::value;
            return run_dgrad<T, F, kDgTH, kTW, kDgMinb>(a, dt, st);
        });
    });
}

int strided_wgrad_slices(const Shape &s, dwconv_dtype dt) {
    if (!covered(s, dt)) return 0;
    const SArgs a = args_of(s);
    int Zc = 0;
    by_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        return by_filter<T>(s.FH, [&](auto f) {
            constexpr int F = decltype(f)::value;
            Geo g;
            size_t smem;
            if (!plan_wgrad<T, F, wgrad_th<T, F>(), kTW, wgrad_minb<T, F>()>(a, g, Zc, smem, false)) Zc = 0;
            return cudaSuccess;
        });
    });
    return Zc;
}

cudaError_t launch_strided_wgrad(const Shape &s, dwconv_dtype dt, const void *x, const void *dy, float *part,
                                 float *dw, cudaStream_t st) {
    if (!covered(s, dt)) return cudaErrorNotSupported;
    SArgs a = args_of(s);
    a.in = x; a.dy = dy;
    return by_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        return by_filter<T>(s.FH, [&](auto f) {
            constexpr int F = decltype(f)::value;
            return run_wgrad<T, F, wgrad_th<T, F>(), kTW, wgrad_minb<T, F>()>(a, dt, part, dw, st);
        });
    });
}

}  // namespace dwc
