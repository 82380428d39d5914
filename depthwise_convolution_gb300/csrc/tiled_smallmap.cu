// Whole-map kernels for small maps: 7x7 inputs with 3x3 / 5x5 / 7x7 filters
// and "same" padding (P = F / 2), stride 1 -- the last stage of the CNNs the
// Flash-DWC evaluation runs (ConvNeXt, RepLKNet: 7x7 maps, 768 channels).
//
// On such maps most taps of a tile-based kernel land in the padding (for 7x7
// filters only 37 of the 49 (output, tap) pairs per axis are inside the map,
// 57 % in 2-D), and tiles sized for large maps compute padding rows too.  Here
// a thread owns one image and one channel pair (one channel for fp32) and walks the whole map with
// the map size and padding known at compile time, so every multiply-add it
// issues is a tap that lands inside the input; no shared memory and no halo:
// a warp's 32 channel pairs of one pixel are one 128-byte load or store.
//
// Forward (and the stride-1 input gradient: the forward pass of dy with the
// filter rotated by 180 degrees, Flash-DWC §5.1; "same" padding maps to
// itself): the thread loads its whole map and its filter into registers (49
// independent loads: one round trip), then for each output row accumulates in
// fp32 (Mac<T>, bias first) and stores the row.  A lane holds a channel pair
// of 16-bit data, or one channel of fp32 data (so that both fit).
//
// Weight gradient (fp32 data; 16-bit data stays on the register-tiled
// tiled_wgrad kernel, measured faster for it: 23.3 against 25.3 us for bf16
// 7x7 on x[128,7,7,768], while fp32 takes 23.4 us here against 78 us on the
// large-filter weight-gradient kernel): CTA = 32 lanes x 4 image slots; each
// thread sums dy * x for every tap over its images (fp32 accumulators for all
// F x F taps, the image's x and dy maps in registers),
// the 4 slots are added in a fixed order through shared memory, the CTA
// writes part[z][tap][c] for its image range z, and wgrad_reduce adds the
// ranges in a fixed order (bit-identical from call to call).
#include "common.cuh"

namespace dwc {
namespace {

constexpr int kMap = 7;   // map height and width
constexpr int kSlots = 4; // warps of a CTA: images (forward) or image slots (weight gradient)
constexpr int kSMThreads = 32 * kSlots;

// What one lane holds per pixel: a packed channel pair for 16-bit data (one
// mixed-precision FMA per channel, fp32 accumulators), one channel for fp32
// data (so that the map and the filter fit in registers).
template <typename T> struct Lane {
    static constexpr int CH = 2;
    using V = typename Mac<T>::V;
    using A = float2;
    static __device__ __forceinline__ V load(const T *p) { return Mac<T>::load(p); }
    static __device__ __forceinline__ void fma(A &acc, V a, V b) { Mac<T>::fma(acc, a, b); }
    static __device__ __forceinline__ A zero() { return make_float2(0.f, 0.f); }
    static __device__ __forceinline__ A bias(const float *b, int c) { return make_float2(b[c], b[c + 1]); }
    static __device__ __forceinline__ void store(T *p, A v) { Pair<T>::store(p, v); }
    static __device__ __forceinline__ void store_f32(float *p, A v) { p[0] = v.x; p[1] = v.y; }
    static __device__ __forceinline__ void add(A &s, A v) { s.x += v.x; s.y += v.y; }
};
template <> struct Lane<float> {
    static constexpr int CH = 1;
    using V = float;
    using A = float;
    static __device__ __forceinline__ V load(const float *p) { return *p; }
    static __device__ __forceinline__ void fma(A &acc, V a, V b) { acc = fmaf(a, b, acc); }
    static __device__ __forceinline__ A zero() { return 0.f; }
    static __device__ __forceinline__ A bias(const float *b, int c) { return b[c]; }
    static __device__ __forceinline__ void store(float *p, A v) { *p = v; }
    static __device__ __forceinline__ void store_f32(float *p, A v) { *p = v; }
    static __device__ __forceinline__ void add(A &s, A v) { s += v; }
};

template <typename T> __host__ __device__ constexpr int lanes_channels() { return 32 * Lane<T>::CH; }  // channels of a warp

// The thread's whole map: 49 independent loads (one round trip), then every
// use comes from registers.
template <typename T>
__device__ __forceinline__ void load_map(const T *img, int C, typename Lane<T>::V (&m)[kMap][kMap]) {
#pragma unroll
    for (int i = 0; i < kMap; ++i)
#pragma unroll
        for (int j = 0; j < kMap; ++j) m[i][j] = Lane<T>::load(img + (i * kMap + j) * C);
}

// CTAs per SM the forward kernel's registers are sized for (16-bit data).
// Measured on GB300 (bf16, x[128,7,7,768]): 3 -> 16.2 us for 7x7 filters,
// 2 -> 17.7, 4 -> 16.9 (the register-tiled tile kernel: 24.8).
#ifndef DWCONV_SM_FWD16_MINB
#define DWCONV_SM_FWD16_MINB 3
#endif

// FUSE (forward only): the BN+Act prologue and the affine+activation epilogue
// of the fused forward pass (Flash-DWC §5.2) -- 1: piecewise-linear
// activations only, 2: all; 0: plain.  The prologue rewrites the thread's
// loaded map in registers (x' = round_T(act(s x + t))); positions outside the
// map are never read, so the padding of x' stays zero as the fusion requires.
template <typename T, int F, int FUSE>
__global__ void __launch_bounds__(kSMThreads, sizeof(T) == 2 ? DWCONV_SM_FWD16_MINB : 3)
    smallmap_fwd_kernel(const T *__restrict__ in, const T *__restrict__ w, const float *__restrict__ bias,
                        T *__restrict__ out, int N, int C, int flip, Fuse fz) {
    constexpr int P = F / 2;
    using L = Lane<T>;
    const int lane = threadIdx.x % 32, slot = threadIdx.x / 32;
    const int c = blockIdx.x * lanes_channels<T>() + L::CH * lane;
    const int n = blockIdx.y * kSlots + slot;
    if (c >= C || n >= N) return;
    typename L::V xr[kMap][kMap], wr[F][F];
    load_map<T>(in + (long long)n * kMap * kMap * C + c, C, xr);
    if constexpr (FUSE > 0) {
        if (fz.pre()) {
            const Affine a0 = affine_in(fz, c);
            if constexpr (L::CH == 2) {
                const Affine a1 = affine_in(fz, c + 1);
                const float2 s2 = make_float2(a0.s, a1.s), t2 = make_float2(a0.t, a1.t);
                with_act<FUSE == 1>(fz.in_act, [&](auto act) {
                    constexpr int A = decltype(act)::value;
#pragma unroll
                    for (int i = 0; i < kMap; ++i)
#pragma unroll
                        for (int j = 0; j < kMap; ++j) xr[i][j] = prologue_packed<T, A>(xr[i][j], s2, t2);
                });
            } else {
                with_act<FUSE == 1>(fz.in_act, [&](auto act) {
                    constexpr int A = decltype(act)::value;
#pragma unroll
                    for (int i = 0; i < kMap; ++i)
#pragma unroll
                        for (int j = 0; j < kMap; ++j) xr[i][j] = activate(fmaf(a0.s, xr[i][j], a0.t), A);
                });
            }
        }
    }
#pragma unroll
    for (int fh = 0; fh < F; ++fh)
#pragma unroll
        for (int fw = 0; fw < F; ++fw) {
            const int sh = flip ? F - 1 - fh : fh, sw = flip ? F - 1 - fw : fw;
            wr[fh][fw] = L::load(w + (sh * F + sw) * C + c);
        }
    const typename L::A b = bias ? L::bias(bias, c) : L::zero();
    T *o = out + (long long)n * kMap * kMap * C + c;
#pragma unroll
    for (int oh = 0; oh < kMap; ++oh) {
        typename L::A acc[kMap];
#pragma unroll
        for (int ow = 0; ow < kMap; ++ow) acc[ow] = b;
#pragma unroll
        for (int fh = 0; fh < F; ++fh) {
            const int ih = oh - P + fh;
            if (ih < 0 || ih >= kMap) continue;
#pragma unroll
            for (int fw = 0; fw < F; ++fw)
#pragma unroll
                for (int ow = 0; ow < kMap; ++ow) {
                    const int iw = ow - P + fw;
                    if (iw < 0 || iw >= kMap) continue;
                    L::fma(acc[ow], wr[fh][fw], xr[ih][iw]);
                }
        }
        if constexpr (FUSE > 0) {
            if (fz.post()) {
                const Affine o0 = affine_out(fz, c);
                const Affine o1 = L::CH == 2 ? affine_out(fz, c + 1) : o0;
                with_act<FUSE == 1>(fz.out_act, [&](auto act) {
                    constexpr int A = decltype(act)::value;
#pragma unroll
                    for (int ow = 0; ow < kMap; ++ow) {
                        if constexpr (L::CH == 2) {
                            acc[ow].x = activate(fmaf(o0.s, acc[ow].x, o0.t), A);
                            acc[ow].y = activate(fmaf(o1.s, acc[ow].y, o1.t), A);
                        } else {
                            acc[ow] = activate(fmaf(o0.s, acc[ow], o0.t), A);
                        }
                    }
                });
            }
        }
#pragma unroll
        for (int ow = 0; ow < kMap; ++ow) L::store(o + (oh * kMap + ow) * C, acc[ow]);
    }
}

template <typename T, int F>
__global__ void __launch_bounds__(kSMThreads, 3)
    smallmap_wgrad_kernel(const T *__restrict__ x, const T *__restrict__ dy, float *__restrict__ part, int N, int C,
                          int per_range) {
    constexpr int P = F / 2;
    using L = Lane<T>;
    __shared__ typename L::A red[kSlots - 1][F * F][32];  // slots 1.. (slot 0 adds from registers)
    const int lane = threadIdx.x % 32, slot = threadIdx.x / 32;
    const int c = blockIdx.x * lanes_channels<T>() + L::CH * lane;
    const int z = blockIdx.y;
    const int n0 = z * per_range, n1 = min(N, n0 + per_range);
    typename L::A acc[F][F];
#pragma unroll
    for (int fh = 0; fh < F; ++fh)
#pragma unroll
        for (int fw = 0; fw < F; ++fw) acc[fh][fw] = L::zero();
    if (c < C) {
        for (int n = n0 + slot; n < n1; n += kSlots) {
            typename L::V xr[kMap][kMap], dr[kMap][kMap];
            load_map<T>(x + (long long)n * kMap * kMap * C + c, C, xr);
            load_map<T>(dy + (long long)n * kMap * kMap * C + c, C, dr);
#pragma unroll
            for (int oh = 0; oh < kMap; ++oh)
#pragma unroll
                for (int fh = 0; fh < F; ++fh) {
                    const int ih = oh - P + fh;
                    if (ih < 0 || ih >= kMap) continue;
#pragma unroll
                    for (int fw = 0; fw < F; ++fw)
#pragma unroll
                        for (int ow = 0; ow < kMap; ++ow) {
                            const int iw = ow - P + fw;
                            if (iw < 0 || iw >= kMap) continue;
                            L::fma(acc[fh][fw], dr[oh][ow], xr[ih][iw]);
                        }
                }
        }
    }
    if (slot > 0) {
#pragma unroll
        for (int fh = 0; fh < F; ++fh)
#pragma unroll
            for (int fw = 0; fw < F; ++fw) red[slot - 1][fh * F + fw][lane] = acc[fh][fw];
    }
    __syncthreads();
    if (slot == 0 && c < C) {
        // Slot 0's sum, then slots 1, 2, 3 in order: a fixed order.
#pragma unroll
        for (int fh = 0; fh < F; ++fh)
#pragma unroll
            for (int fw = 0; fw < F; ++fw) {
                typename L::A s = acc[fh][fw];
#pragma unroll
                for (int q = 0; q < kSlots - 1; ++q) L::add(s, red[q][fh * F + fw][lane]);
                L::store_f32(part + ((long long)z * F * F + fh * F + fw) * C + c, s);
            }
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

template <typename Fn>
cudaError_t by_filter(int F, Fn &&fn) {
    switch (F) {
        case 3: return fn(std::integral_constant<int, 3>{});
        case 5: return fn(std::integral_constant<int, 5>{});
        case 7: return fn(std::integral_constant<int, 7>{});
        default: return cudaErrorNotSupported;
    }
}

// 7x7 map, square odd filter, "same" padding, unit stride and dilation on the
// whole tensor, fp32 / fp16 / bf16, even channel count.
int channels_per_cta(dwconv_dtype dt) { return dt == DWCONV_FP32 ? lanes_channels<float>() : lanes_channels<__half>(); }

// The shapes the whole-map kernels take (any fusion aside).
bool covered_shape(const TiledConv &p, dwconv_dtype dt) {
    const int F = p.FH;
    return (dt == DWCONV_FP32 || dt == DWCONV_FP16 || dt == DWCONV_BF16) && p.FW == F &&
           (F == 3 || F == 5 || F == 7) && p.pad_h == F / 2 && p.pad_w == F / 2 && p.Hs == kMap &&
           p.Ws == kMap && p.Hf == kMap && p.Wf == kMap && p.in_step_h == 1 && p.in_step_w == 1 &&
           p.in_off_h == 0 && p.in_off_w == 0 && p.OHs == kMap && p.OWs == kMap && p.OHf == kMap &&
           p.OWf == kMap && p.out_step_h == 1 && p.out_step_w == 1 && !p.zero_phases && !p.transpose &&
           p.C % 2 == 0;
}
bool covered(const TiledConv &p, dwconv_dtype dt) { return covered_shape(p, dt) && !p.fz.pre() && !p.fz.post(); }

// Image ranges of the weight gradient: about two waves of CTAs over the
// channel groups, at least one image per slot; a pure function of the shape
// (launch = false: the workspace bound) or of the device (launch = true).
int wgrad_ranges(const TiledConv &p, bool launch, int *per_range) {
    const long long groups = (p.C + 63) / 64;  // channel groups of the 16-bit kernels (the fp32 ones have 2x)
    long long z = (2LL * plan_sms(launch) + groups - 1) / groups;
    z = std::max(1LL, std::min<long long>(z, (p.N + kSlots - 1) / kSlots));
    const int per = (int)((p.N + z - 1) / z);
    *per_range = per;
    return (int)((p.N + per - 1) / per);
}

}  // namespace

cudaError_t launch_smallmap(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (!covered_shape(p, dt)) return cudaErrorNotSupported;
    const bool fused = p.fz.pre() || p.fz.post();
    if (fused && p.flip) return cudaErrorNotSupported;  // fusion is a forward-pass feature
    const int level = !fused ? 0 : act_is_light(p.fz.in_act) && act_is_light(p.fz.out_act) ? 1 : 2;
    const int cpc = channels_per_cta(dt);
    const dim3 grid((unsigned)((p.C + cpc - 1) / cpc), (unsigned)((p.N + kSlots - 1) / kSlots));
    return by_dtype(dt, [&](auto tag) {
        using T = decltype(tag);
        return by_filter(p.FH, [&](auto f) {
            constexpr int F = decltype(f)::value;
            auto go = [&](auto fuse) {
                smallmap_fwd_kernel<T, F, decltype(fuse)::value><<<grid, kSMThreads, 0, st>>>(
                    static_cast<const T *>(p.in), static_cast<const T *>(p.w), p.bias, static_cast<T *>(p.out),
                    p.N, p.C, p.flip, p.fz);
            };
            if (level == 0) go(std::integral_constant<int, 0>{});
            else if (level == 1) go(std::integral_constant<int, 1>{});
            else go(std::integral_constant<int, 2>{});
            note_launches(1);
            note_kernel("smallmap");
            return cudaGetLastError();
        });
    });
}

int smallmap_wgrad_slices(const TiledConv &p, dwconv_dtype dt) {
    if (dt != DWCONV_FP32 || !covered(p, dt)) return 0;
    int per = 0;
    return wgrad_ranges(p, false, &per);
}

cudaError_t launch_smallmap_wgrad(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st) {
    if (dt != DWCONV_FP32 || !covered(p, dt)) return cudaErrorNotSupported;
    int per = 0;
    const int Z = wgrad_ranges(p, true, &per);
    const int cpc = channels_per_cta(dt);
    const dim3 grid((unsigned)((p.C + cpc - 1) / cpc), (unsigned)Z);
    cudaError_t e = by_filter(p.FH, [&](auto f) {
        constexpr int F = decltype(f)::value;
        smallmap_wgrad_kernel<float, F><<<grid, kSMThreads, 0, st>>>(
            static_cast<const float *>(p.in), static_cast<const float *>(p.dy), part, p.N, p.C, per);
        note_launches(1);
        note_kernel("smallmap_wgrad");
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;
    return launch_wgrad_reduce(part, Z, (long long)p.FH * p.FW * p.C, static_cast<float *>(p.out), st);
}

}  // namespace dwc
