// Register-tiled weight gradient for large filters (FW >= 8 in the kernel's
// view, any FH; strips taller than wide arrive transposed), all float dtypes.
//
//   dw[fh,fw,c] = sum over (n, i, j) of dy[n,i,j,c] * x_sub[n, i - pad_h + fh, j - pad_w + fw, c]
//
// The FH x FW accumulators of a channel no longer fit in one thread, so the
// taps are tiled over threads (Flash-DWC §5.1 "BFC" with the accumulation-axis
// split; the tap tiling plays the role §5.1 gives the flexible TM tiles):
//   * CTA = 16 channel pairs x 16 tap tiles of THF x TWF taps (256 threads);
//     the tap tiles form a tap group of RTT*THF rows x CTT*TWF columns,
//     CTT = 1, 2 or 4 by the filter width, RTT = 16/CTT (fewer for short
//     filters, the other tiles idle);
//   * grid = channel tiles x slices Zc x tap groups; CTA (ctile, z, group)
//     takes the work units z, z + Zc, ... of its channel tile, a unit being
//     OTH x OTW dy positions of one image.  Per unit one thread stages, with
//     two TMA tensor copies on one mbarrier, the dy tile and the x halo the
//     tap group reads ((OTH + GH - 1) x (OTW + GW - 1), zeros outside the
//     input), double-buffered with bounded waits;
//   * a thread walks the dy tile row by row; for each of its THF filter rows
//     it slides a TWF-wide register window along the x row (one new value per
//     dy column), and every dy value it reads feeds THF * TWF multiply-adds
//     into fp32 accumulators that live for the whole CTA;
//   * each (channel pair, tap) belongs to one thread of the CTA, so the CTA
//     writes part[z][tap][c] directly; wgrad_reduce (direct.cu) sums the Zc
//     slices in a fixed order (bit-identical from call to call).
#include <algorithm>

#include "tiled_common.cuh"

namespace dwc {
namespace {

using namespace tiled;

constexpr int kWLThreads = 256;
constexpr int kTapTiles = kWLThreads / kPairs;  // 16
constexpr int kTHF = 2, kTWF = 8;               // taps per thread: filter rows x filter columns
constexpr int kOTH = 8;                         // dy rows per unit

constexpr int kOTW = 16;                        // dy columns per unit

struct GeoW {
    int CTT, RTT;          // tap tiles per group: columns x rows (product 16)
    int GH, GW;            // taps per group: rows, columns
    int groups_h, groups_w, groups;
    int HH, HW;            // x halo rows, columns per unit
    int tiles_h, tiles_w;  // units along dy rows / columns
    int per_ctile, ctiles;
    unsigned x_bytes, dy_bytes, stage;  // box bytes, bytes of one pipeline stage
};

inline GeoW make_geo_w(const TiledConv &p, size_t es) {
    constexpr int OTW = kOTW;
    GeoW g{};
    const int cols = (p.FW + kTWF - 1) / kTWF;
    g.CTT = cols >= 4 ? 4 : cols >= 2 ? 2 : 1;
    // No more tap-tile rows than the filter has (short filters leave tiles idle
    // rather than stage halo rows no tap reads).
    g.RTT = std::min(kTapTiles / g.CTT, (p.FH + kTHF - 1) / kTHF);
    g.GH = g.RTT * kTHF;
    g.GW = g.CTT * kTWF;
    g.groups_h = (p.FH + g.GH - 1) / g.GH;
    g.groups_w = (p.FW + g.GW - 1) / g.GW;
    g.groups = g.groups_h * g.groups_w;
    g.HH = kOTH + g.GH - 1;
    g.HW = OTW + g.GW - 1;
    g.tiles_h = (p.OHs + kOTH - 1) / kOTH;
    g.tiles_w = (p.OWs + OTW - 1) / OTW;
    g.ctiles = (p.C + 31) / 32;
    const long long per = (long long)p.N * g.tiles_h * g.tiles_w;
    g.per_ctile = per < (1LL << 30) ? (int)per : 0;
    g.x_bytes = (unsigned)((size_t)g.HH * g.HW * 32 * es);
    g.dy_bytes = (unsigned)((size_t)kOTH * OTW * 32 * es);
    g.stage = align128(g.x_bytes) + align128(g.dy_bytes);
    return g;
}

template <typename T>
__global__ void __launch_bounds__(kWLThreads, 1)
    tiled_wgrad_large_kernel(const __grid_constant__ CUtensorMap halo_map, const __grid_constant__ CUtensorMap dy_map,
                             TiledConv p, GeoW g, float *__restrict__ part, int Zc, unsigned *err) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2];
    using M = Mac<T>;
    using V = typename M::V;

    const int tid = threadIdx.x;
    const int cp = tid % kPairs, tt = tid / kPairs;
    const int rtt = tt / g.CTT, ctt = tt % g.CTT;
    const bool active = rtt < g.RTT;  // a tap tile of the group (else idle, barriers only)
    const int grp = blockIdx.x % g.groups;
    const int z = (blockIdx.x / g.groups) % Zc;
    const int ctile = blockIdx.x / (g.groups * Zc);
    const int gh0 = (grp / g.groups_w) * g.GH, gw0 = (grp % g.groups_w) * g.GW;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    // Unit v of the channel tile: dy rows band*OTH.., columns twi*OTW.. of image n.
    auto issue = [&](int v, int b) {
        const int band = v % g.tiles_h, rest = v / g.tiles_h;
        const int twi = rest % g.tiles_w, n = rest / g.tiles_w;
        unsigned char *dst = smem_raw + b * g.stage;
        mbar_arrive_expect_tx(&bars[b], g.x_bytes + g.dy_bytes);
        tma_load_4d(dst, &halo_map, ctile * 32, twi * kOTW - p.pad_w + gw0, band * kOTH - p.pad_h + gh0, n,
                    &bars[b]);
        tma_load_4d(dst + align128(g.x_bytes), &dy_map, ctile * 32, twi * kOTW, band * kOTH, n, &bars[b]);
    };

    float2 acc[kTHF][kTWF];
#pragma unroll
    for (int th = 0; th < kTHF; ++th)
#pragma unroll
        for (int f = 0; f < kTWF; ++f) acc[th][f] = make_float2(0.f, 0.f);

    int v = z;
    if (tid == 0 && v < g.per_ctile) issue(v, 0);
    for (int k = 0; v < g.per_ctile; ++k, v += Zc) {
        const int vn = v + Zc;
        if (tid == 0 && vn < g.per_ctile) issue(vn, (k + 1) & 1);
        if (!mbar_wait(&bars[k & 1], (k >> 1) & 1)) {
            // Give up: record it, let the copy still in flight land, and leave.
            report_timeout(err);
            if (tid == 0 && vn < g.per_ctile) mbar_wait(&bars[(k + 1) & 1], ((k + 1) >> 1) & 1);
            return;
        }
        const unsigned char *cur = smem_raw + (k & 1) * g.stage;
        const T *sx = reinterpret_cast<const T *>(cur) + (rtt * kTHF * g.HW + ctt * kTWF) * 32 + 2 * cp;
        const T *sd = reinterpret_cast<const T *>(cur + align128(g.x_bytes)) + 2 * cp;
        for (int i = 0; active && i < kOTH; ++i) {
            // Window slot s holds x column j + ((s - j) mod TWF) of each of the
            // thread's filter rows; dy column j meets columns j .. j + TWF - 1.
            V xw[kTHF][kTWF];
            const T *xr[kTHF];
#pragma unroll
            for (int th = 0; th < kTHF; ++th) {
                xr[th] = sx + (i + th) * g.HW * 32;
#pragma unroll
                for (int f = 0; f < kTWF; ++f) xw[th][f] = M::load(xr[th] + f * 32);
            }
            const T *dr = sd + i * kOTW * 32;
#pragma unroll
            for (int j = 0; j < kOTW; ++j) {
                const V d = M::load(dr + j * 32);
#pragma unroll
                for (int th = 0; th < kTHF; ++th)
#pragma unroll
                    for (int f = 0; f < kTWF; ++f) M::fma(acc[th][f], d, xw[th][(j + f) % kTWF]);
                if (j + 1 < kOTW) {
#pragma unroll
                    for (int th = 0; th < kTHF; ++th) xw[th][j % kTWF] = M::load(xr[th] + (j + kTWF) * 32);
                }
            }
        }
        __syncthreads();  // this buffer is refilled by the copy issued next iteration
    }

    // Every (channel pair, tap) of the CTA belongs to this thread alone.
    const int c = ctile * 32 + 2 * cp;
    if (!active || c >= p.C) return;
#pragma unroll
    for (int th = 0; th < kTHF; ++th)
#pragma unroll
        for (int f = 0; f < kTWF; ++f) {
            const int fh = gh0 + rtt * kTHF + th, fw = gw0 + ctt * kTWF + f;
            if (fh >= p.FH || fw >= p.FW) continue;
            const int tap = p.transpose ? fw * p.FH + fh : fh * p.FW + fw;  // memory order
            float *dst = part + ((long long)z * p.FH * p.FW + tap) * p.C + c;
            dst[0] = acc[th][f].x;
            dst[1] = acc[th][f].y;
        }
}

// Plan: geometry and the slice count Zc (about two CTAs per SM for 16-bit
// data, one for fp32, over all channel tiles and tap groups), for the
// workspace bound or the current device (plan_sms).  Returns false if no
// instance covers the shape.
bool plan_w(const TiledConv &p, dwconv_dtype dt, GeoW &g, int &Zc, bool launch) {
    if (dt != DWCONV_FP32 && dt != DWCONV_FP16 && dt != DWCONV_BF16) return false;
    const size_t es = dt == DWCONV_FP32 ? 4 : 2;
    g = make_geo_w(p, es);
    if (g.per_ctile == 0 || g.HH > 256 || g.HW > 256 || 2 * (size_t)g.stage > 220 * 1024) return false;
    const long long target = (long long)plan_sms(launch) * (es == 2 ? 2 : 1);
    long long z = target / ((long long)g.ctiles * g.groups);
    if (z > g.per_ctile) z = g.per_ctile;
    if (z < 1) z = 1;
    if ((long long)g.ctiles * g.groups * z >= (1LL << 31)) return false;
    Zc = (int)z;
    return true;
}

template <typename T>
cudaError_t run_w(const TiledConv &p, dwconv_dtype dt, const GeoW &g, int Zc, float *part, cudaStream_t st) {
    const size_t es = sizeof(T);
    // x: the taps' sub-grid of p.in, one box = one unit's halo for one tap group.
    const char *base = static_cast<const char *>(p.in) + ((size_t)p.in_off_h * p.Wf + p.in_off_w) * p.C * es;
    const uint64_t dims[4] = {(uint64_t)p.C, (uint64_t)p.Ws, (uint64_t)p.Hs, (uint64_t)p.N};
    uint64_t str[3];
    in_strides(p, es, str);
    const uint32_t box[4] = {32, (uint32_t)g.HW, (uint32_t)g.HH, 1};
    // dy [N][OH][OW][C] in memory; OHs x OWs in the kernel's orientation.
    const uint64_t ddims[4] = {(uint64_t)p.C, (uint64_t)p.OWs, (uint64_t)p.OHs, (uint64_t)p.N};
    const uint64_t mem_row = (uint64_t)(p.transpose ? p.OHs : p.OWs) * p.C * es, mem_col = (uint64_t)p.C * es;
    const uint64_t dstr[3] = {p.transpose ? mem_row : mem_col, p.transpose ? mem_col : mem_row,
                              (uint64_t)p.OHs * p.OWs * p.C * es};
    const uint32_t dbox[4] = {32, (uint32_t)kOTW, (uint32_t)kOTH, 1};
    CUtensorMap halo_map, dy_map;
    if (!encode_tmap_4d(&halo_map, dt, base, dims, str, box) || !encode_tmap_4d(&dy_map, dt, p.dy, ddims, dstr, dbox))
        return cudaErrorNotSupported;
    const size_t smem = 2 * (size_t)g.stage;
    auto kern = tiled_wgrad_large_kernel<T>;
    cudaError_t e = kernel_setup(reinterpret_cast<const void *>(kern), kWLThreads, smem, nullptr);
    if (e != cudaSuccess) return e;
    kern<<<g.ctiles * g.groups * Zc, kWLThreads, smem, st>>>(halo_map, dy_map, p, g, part, Zc, device_error_word());
    note_launches(1);
    note_kernel("tiled_wgrad_large");
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_wgrad_reduce(part, Zc, (long long)p.FH * p.FW * p.C, static_cast<float *>(p.out), st);
}

}  // namespace

int tiled_wgrad_large_slices(const TiledConv &p, dwconv_dtype dt) {
    GeoW g;
    int Zc = 0;
    return plan_w(p, dt, g, Zc, false) ? Zc : 0;
}

cudaError_t launch_tiled_wgrad_large(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st) {
    GeoW g;
    int Zc = 0;
    if (!plan_w(p, dt, g, Zc, true)) return cudaErrorNotSupported;
    switch (dt) {
        case DWCONV_FP32: return run_w<float>(p, dt, g, Zc, part, st);
        case DWCONV_FP16: return run_w<__half>(p, dt, g, Zc, part, st);
        case DWCONV_BF16: return run_w<__nv_bfloat16>(p, dt, g, Zc, part, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
