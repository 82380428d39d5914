// Internal declarations shared by the libdwconv translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "dwconv.h"

namespace dwc {

// Problem geometry after validation.  H, W, C are input sizes; OH, OW the
// forward output sizes (floor convention).
struct Shape {
    int N, H, W, C, FH, FW;
    int SH, SW, DH, DW, PH, PW;  // stride, dilation, padding per axis
    int OH, OW;
};

// Counts kernel launches for dwconv_launch_count().
void note_launches(int n);
// Records the kernel family of the calling thread's latest pass for
// dwconv_last_kernel() (a static string).
void note_kernel(const char *family);

// Number of SMs of the current device (cached per device).
int sm_count();

// Prepares `kern` for a launch of `threads` threads with `smem` bytes of
// dynamic shared memory: raises its shared-memory limit if this context has
// not set one that large yet (the limit is per kernel and is never lowered)
// and, if per_sm is not null, stores how many such CTAs fit on an SM (looked
// up once per kernel, context, block size and shared-memory size), so a
// repeated launch pays table lookups instead of two runtime queries.
cudaError_t kernel_setup(const void *kern, int threads, size_t smem, int *per_sm);

// SM count and shared memory per SM that a split-reduction plan is sized for.
// Workspace sizes are pure functions of the shape, so they are planned for an
// upper bound (kPlanMaxSms SMs: sm_103a parts have at most 160; 228 KB of
// shared memory per SM); a launch plans for the current device, capped at
// those bounds, so the slices it writes never outnumber the ones its
// workspace was sized for.
constexpr int kPlanMaxSms = 160;
constexpr int kPlanMaxSmemPerSm = 228 * 1024;
int plan_sms(bool launch);
int plan_smem_per_sm(bool launch);

// ---- element access --------------------------------------------------------

// Two adjacent channels of one storage type, widened to / narrowed from float2.
template <typename T> struct Pair;

template <> struct Pair<float> {
    static __device__ __forceinline__ float2 load(const float *p) {
        return *reinterpret_cast<const float2 *>(p);
    }
    static __device__ __forceinline__ void store(float *p, float2 v) {
        *reinterpret_cast<float2 *>(p) = v;
    }
};

template <> struct Pair<__half> {
    static __device__ __forceinline__ float2 load(const __half *p) {
        return __half22float2(*reinterpret_cast<const __half2 *>(p));
    }
    static __device__ __forceinline__ void store(__half *p, float2 v) {
        *reinterpret_cast<__half2 *>(p) = __float22half2_rn(v);
    }
};

template <> struct Pair<__nv_bfloat16> {
    static __device__ __forceinline__ float2 load(const __nv_bfloat16 *p) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float2 v) {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __float22bfloat162_rn(v);
    }
};

// FP8 E4M3 (inputs of the forward pass only): a pair widens exactly to two
// floats (through f16, which holds every E4M3 value); the store rounds to
// nearest even with saturation at +-448 (used only by code paths the host
// never selects for FP8, kept so that the templates compile).
template <> struct Pair<__nv_fp8_e4m3> {
    static __device__ __forceinline__ float2 load(const __nv_fp8_e4m3 *p) {
        const __half2_raw h =
            __nv_cvt_fp8x2_to_halfraw2(*reinterpret_cast<const __nv_fp8x2_storage_t *>(p), __NV_E4M3);
        return __half22float2(*reinterpret_cast<const __half2 *>(&h));
    }
    static __device__ __forceinline__ void store(__nv_fp8_e4m3 *p, float2 v) {
        *reinterpret_cast<__nv_fp8x2_storage_t *>(p) = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
    }
};

// Output element type of the forward pass per input type: FP8 inputs give
// bf16 outputs, every other type its own.
template <typename T> struct OutOf { using type = T; };
template <> struct OutOf<__nv_fp8_e4m3> { using type = __nv_bfloat16; };
// Tensor-core operand type per input type: FP8 E4M3 converts exactly to f16.
template <typename T> struct MmaIn { using type = T; };
template <> struct MmaIn<__nv_fp8_e4m3> { using type = __half; };

// Multiply-accumulate on a channel pair, per storage type.  A pair is held in
// registers as it is stored: fp32 data as float2, 16-bit data as one packed
// 32-bit word.  fp32 uses the packed fma.rn.f32x2; 16-bit data uses the
// sm_100+ mixed-precision fma.rn.f32.{f16,bf16}, whose 16 x 16-bit product is
// exact in fp32 and is added to the fp32 accumulator with one rounding -- the
// same result as widening first and using an fp32 FMA, without the widening
// instructions.
template <typename T> struct Mac;

template <> struct Mac<float> {
    using V = float2;
    static __device__ __forceinline__ V load(const float *p) { return *reinterpret_cast<const float2 *>(p); }
    static __device__ __forceinline__ V zero() { return make_float2(0.f, 0.f); }
    static __device__ __forceinline__ void fma(float2 &acc, V a, V b) { acc = __ffma2_rn(a, b, acc); }
};

template <> struct Mac<__half> {
    using V = unsigned;
    static __device__ __forceinline__ V load(const __half *p) { return *reinterpret_cast<const unsigned *>(p); }
    static __device__ __forceinline__ V zero() { return 0u; }
    static __device__ __forceinline__ void fma(float2 &acc, V a, V b) {
        asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %2;\n mov.b32 {bl, bh}, %3;\n"
            " fma.rn.f32.f16 %0, al, bl, %0;\n fma.rn.f32.f16 %1, ah, bh, %1;\n}\n"
            : "+f"(acc.x), "+f"(acc.y)
            : "r"(a), "r"(b));
    }
};

template <> struct Mac<__nv_bfloat16> {
    using V = unsigned;
    static __device__ __forceinline__ V load(const __nv_bfloat16 *p) {
        return *reinterpret_cast<const unsigned *>(p);
    }
    static __device__ __forceinline__ V zero() { return 0u; }
    static __device__ __forceinline__ void fma(float2 &acc, V a, V b) {
        asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %2;\n mov.b32 {bl, bh}, %3;\n"
            " fma.rn.f32.bf16 %0, al, bl, %0;\n fma.rn.f32.bf16 %1, ah, bh, %1;\n}\n"
            : "+f"(acc.x), "+f"(acc.y)
            : "r"(a), "r"(b));
    }
};

// FP8: a pair converts exactly to a packed f16 pair on load (one cvt), then
// the mixed-precision FMAs of the f16 path.
template <> struct Mac<__nv_fp8_e4m3> {
    using V = unsigned;
    static __device__ __forceinline__ V load(const __nv_fp8_e4m3 *p) {
        const __half2_raw h =
            __nv_cvt_fp8x2_to_halfraw2(*reinterpret_cast<const __nv_fp8x2_storage_t *>(p), __NV_E4M3);
        return *reinterpret_cast<const unsigned *>(&h);
    }
    static __device__ __forceinline__ V zero() { return 0u; }
    static __device__ __forceinline__ void fma(float2 &acc, V a, V b) { Mac<__half>::fma(acc, a, b); }
};

// Widening variant: a channel pair is widened to float2 when loaded and every
// multiply-add is one packed fma.rn.f32x2 (the same products and roundings as
// Mac<T>; fewer FMA instructions per value, at the cost of the conversions
// and twice the registers per held value).
template <typename T> struct MacW {
    using V = float2;
    static __device__ __forceinline__ V load(const T *p) { return Pair<T>::load(p); }
    static __device__ __forceinline__ V zero() { return make_float2(0.f, 0.f); }
    static __device__ __forceinline__ void fma(float2 &acc, V a, V b) { acc = __ffma2_rn(a, b, acc); }
};

// Scalar widening / rounding (round to nearest even for 16-bit outputs).
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__nv_fp8_e4m3 v) { return float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __nv_fp8_e4m3 from_f32<__nv_fp8_e4m3>(float v) { return __nv_fp8_e4m3(v); }

// ---- fused BN+Act prologue / affine+activation epilogue ---------------------

// Flash-DWC §5.2 "Kernel fusion": per channel c, the forward pass may read
//   x' = round_T(act_in(in_scale[c] * x + in_shift[c]))   at every input position
// (the zero padding applies to x') and write
//   y = round_T(act_out(out_scale[c] * (conv + bias[c]) + out_shift[c])).
// Null scale = 1, null shift = 0, act 0 = identity; fp32 arithmetic, one
// fmaf for the affine map.
struct Fuse {
    const float *in_scale, *in_shift;
    int in_act;
    const float *out_scale, *out_shift;
    int out_act;
    __host__ __device__ bool pre() const { return in_scale || in_shift || in_act; }
    __host__ __device__ bool post() const { return out_scale || out_shift || out_act; }
};

// Gauss error function for GELU, from Abramowitz & Stegun, "Handbook of
// Mathematical Functions", formula 7.1.26: for x >= 0,
//   erfc(x) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2) + e(x),
//   t = 1 / (1 + p x),  |e(x)| <= 1.5e-7,
// with p and a1..a5 as printed there.  Evaluated in fp32 with the fast
// exponential and reciprocal (a few fp32 ulps more).
__device__ __forceinline__ float erfc_as(float x) {
    const float t = __fdividef(1.f, fmaf(0.3275911f, x, 1.f));
    float q = fmaf(1.061405429f, t, -1.453152027f);
    q = fmaf(q, t, 1.421413741f);
    q = fmaf(q, t, -0.284496736f);
    q = fmaf(q, t, 0.254829592f);
    return q * t * __expf(-x * x);
}

// v * Phi(v), Phi the standard normal distribution function:
// Phi(v) = erfc(-v / sqrt 2) / 2, i.e. 1 - erfc(|v| / sqrt 2) / 2 for v >= 0
// and erfc(|v| / sqrt 2) / 2 for v < 0 (no cancellation in the negative tail).
__device__ __forceinline__ float gelu_erf(float v) {
    const float h = 0.5f * erfc_as(fabsf(v) * 0.7071067811865476f);
    return v * (v >= 0.f ? 1.f - h : h);
}

__device__ __forceinline__ float activate(float v, int act) {
    switch (act) {
        case DWCONV_ACT_RELU: return fmaxf(v, 0.f);
        case DWCONV_ACT_RELU6: return fminf(fmaxf(v, 0.f), 6.f);
        case DWCONV_ACT_SILU: return __fdividef(v, 1.f + __expf(-v));  // v * sigmoid(v)
        case DWCONV_ACT_GELU: return gelu_erf(v);
        default: return v;
    }
}

// Per-channel coefficients of one affine map (channel c must be valid).
struct Affine {
    float s, t;
};
__device__ __forceinline__ Affine affine_in(const Fuse &f, int c) {
    return {f.in_scale ? __ldg(f.in_scale + c) : 1.f, f.in_shift ? __ldg(f.in_shift + c) : 0.f};
}
__device__ __forceinline__ Affine affine_out(const Fuse &f, int c) {
    return {f.out_scale ? __ldg(f.out_scale + c) : 1.f, f.out_shift ? __ldg(f.out_shift + c) : 0.f};
}
__device__ __forceinline__ float apply(Affine a, float v, int act) { return activate(fmaf(a.s, v, a.t), act); }

// Calls f(std::integral_constant<int, act>{}) so that loops over many values
// see the activation as a compile-time constant (one branch per loop, not per
// value).
// With LIGHT, only the piecewise-linear activations (none, ReLU, ReLU6) are
// compiled in: for instances the host calls with no other.
template <bool LIGHT = false, typename F>
__device__ __forceinline__ void with_act(int act, F &&f) {
    switch (act) {
        case DWCONV_ACT_RELU: f(std::integral_constant<int, DWCONV_ACT_RELU>{}); break;
        case DWCONV_ACT_RELU6: f(std::integral_constant<int, DWCONV_ACT_RELU6>{}); break;
        case DWCONV_ACT_SILU:
            if constexpr (!LIGHT) f(std::integral_constant<int, DWCONV_ACT_SILU>{});
            break;
        case DWCONV_ACT_GELU:
            if constexpr (!LIGHT) f(std::integral_constant<int, DWCONV_ACT_GELU>{});
            break;
        default: f(std::integral_constant<int, DWCONV_ACT_NONE>{}); break;
    }
}
__host__ __device__ inline bool act_is_light(int act) {
    return act == DWCONV_ACT_NONE || act == DWCONV_ACT_RELU || act == DWCONV_ACT_RELU6;
}

// A channel pair of a 16-bit type packed in one 32-bit word <-> float2.
template <typename T> __device__ __forceinline__ float2 unpack2(unsigned v);
template <> __device__ __forceinline__ float2 unpack2<__half>(unsigned v) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&v));
}
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(unsigned v) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v));
}
template <typename T> __device__ __forceinline__ unsigned pack2(float2 v);
template <> __device__ __forceinline__ unsigned pack2<__half>(float2 v) {
    const __half2 h = __float22half2_rn(v);
    return *reinterpret_cast<const unsigned *>(&h);
}
template <> __device__ __forceinline__ unsigned pack2<__nv_bfloat16>(float2 v) {
    const __nv_bfloat162 h = __float22bfloat162_rn(v);
    return *reinterpret_cast<const unsigned *>(&h);
}

// Packed max(v, 0) and min(v, 6) on a pair of 16-bit values.  Rounding is
// monotonic and 0 and 6 are exact in both formats, so clamping after the
// rounding gives the rounding of the clamped fp32 value.
template <typename T> __device__ __forceinline__ unsigned clamp_packed(unsigned v, bool six);
template <> __device__ __forceinline__ unsigned clamp_packed<__half>(unsigned v, bool six) {
    __half2 h = __hmax2(*reinterpret_cast<const __half2 *>(&v), __float2half2_rn(0.f));
    if (six) h = __hmin2(h, __float2half2_rn(6.f));
    return *reinterpret_cast<const unsigned *>(&h);
}
template <> __device__ __forceinline__ unsigned clamp_packed<__nv_bfloat16>(unsigned v, bool six) {
    __nv_bfloat162 h = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v), __float2bfloat162_rn(0.f));
    if (six) h = __hmin2(h, __float2bfloat162_rn(6.f));
    return *reinterpret_cast<const unsigned *>(&h);
}

// BN+Act prologue on a packed pair of 16-bit values x: round_T(act(s x + t))
// per half (s, t per half), the affine map as one packed fp32 FMA.
template <typename T, int A>
__device__ __forceinline__ unsigned prologue_packed(unsigned v, float2 s, float2 t) {
    float2 f = __ffma2_rn(unpack2<T>(v), s, t);
    if constexpr (A == DWCONV_ACT_SILU || A == DWCONV_ACT_GELU) {
        f.x = activate(f.x, A);
        f.y = activate(f.y, A);
    }
    unsigned r = pack2<T>(f);
    if constexpr (A == DWCONV_ACT_RELU || A == DWCONV_ACT_RELU6) r = clamp_packed<T>(r, A == DWCONV_ACT_RELU6);
    return r;
}

// The same on an fp32 pair.
template <int A>
__device__ __forceinline__ float2 prologue_f32(float2 v, float2 s, float2 t) {
    float2 f = __ffma2_rn(v, s, t);
    f.x = activate(f.x, A);
    f.y = activate(f.y, A);
    return f;
}

// ---- launchers (each returns the launch's cudaError_t) -----------------------

// Direct kernels: any shape, any dtype the pass supports; one thread per output.
cudaError_t launch_fwd_direct(const Shape &s, dwconv_dtype dt, const void *x, const void *w,
                              const void *bias, void *y, const Fuse &fz, cudaStream_t st);
cudaError_t launch_dgrad_direct(const Shape &s, dwconv_dtype dt, const void *dy, const void *w,
                                void *dx, cudaStream_t st);
// wgrad, first pass: partial sums over Z slices of the N*OH*OW axis into
// part[Z][FH*FW][C]; second pass: fixed-order sum over the Z slices into dw.
cudaError_t launch_wgrad_direct(const Shape &s, dwconv_dtype dt, const void *x, const void *dy,
                                float *part, int Z, cudaStream_t st);
cudaError_t launch_wgrad_reduce(const float *part, int Z, long long count, float *dw,
                                cudaStream_t st);
// Bias gradient, first pass: part[z][c] = sum of dy over the positions of
// slice z of the P = N*OH*OW positions (the second pass is launch_wgrad_reduce
// with count = C).  bias_slices(P, C, false) is a pure function of the shape
// (the workspace size); a launch uses bias_slices(P, C, true) <= that.
int bias_slices(long long P, int C, bool launch);
cudaError_t launch_bias_slices(long long P, int C, dwconv_dtype dt, const void *dy, float *part, int Z,
                               cudaStream_t st);

// Register-tiled kernels for small filters (the whole filter of a channel pair
// held in registers).  The sub-grid description lets one kernel serve the
// forward pass (including stride = dilation cases that read one phase of the
// input) and the phase-decomposed input gradient.
struct TiledConv {
    const void *in;        // x (forward) or dy (input gradient)
    const void *w;
    const float *bias;     // nullable; forward only
    void *out;             // y or dx (dw, float, for the weight gradient)
    const void *dy;        // weight gradient only: dy [N][OHs][OWs][C]
    int N, C;
    int FH, FW;
    int flip;              // 1: filter rotated by 180 degrees
    // Input tensor [N][Hf][Wf][C]; taps read its sub-grid
    //   (in_off_h + in_step_h*i, in_off_w + in_step_w*j), 0 <= i < Hs, 0 <= j < Ws.
    int Hf, Wf, Hs, Ws, in_step_h, in_step_w, in_off_h, in_off_w;
    int pad_h, pad_w;      // sub-grid input row of output row i, tap fh: i - pad_h + fh (cols alike)
    // Output tensor [N][OHf][OWf][C]; computed element (i, j) of the OHs x OWs
    // grid goes to (out_off_h + out_step_h*i, out_off_w + out_step_w*j).  With
    // zero_phases, the other positions of each out_step_h x out_step_w block
    // are written with zeros.
    int OHf, OWf, OHs, OWs, out_step_h, out_step_w, out_off_h, out_off_w, zero_phases;
    Fuse fz;               // forward only; all null / zero: plain convolution
    int half_accumulate;   // weight gradient, fp16 data: fp16 partial sums per unit (opt-in)
    // Transposed view (strip filters taller than wide): the kernel's rows are
    // the tensors' columns.  Hs, Ws, pad_h, pad_w, FH, FW, OHs, OWs are then
    // given in the kernel's orientation (swapped); Hf, Wf, in_step_*, in_off_*,
    // OHf, OWf, out_step_*, out_off_* keep describing memory, and w stays
    // [FH_mem][FW_mem][C] = [FW][FH][C] of the kernel.  Only the large-filter
    // kernels (tiled_large.cu, tiled_mma_large.cu) accept it.
    int transpose;
};

// Byte strides of the taps' input sub-grid along the kernel's columns, rows and
// images (the memory rows and columns exchange roles under p.transpose).
inline void in_strides(const TiledConv &p, size_t es, uint64_t str[3]) {
    const uint64_t col = (uint64_t)p.in_step_w * p.C * es, row = (uint64_t)p.in_step_h * p.Wf * p.C * es;
    str[0] = p.transpose ? row : col;
    str[1] = p.transpose ? col : row;
    str[2] = (uint64_t)p.Hf * p.Wf * p.C * es;
}

// Returns cudaErrorNotSupported when no tiled instance covers the request.
cudaError_t launch_tiled_small(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);

// Tensor-core (mma.sync) forward and input gradient for 16-bit data, 3x3 /
// 5x5 / 7x7 filters, maps more than 8 columns wide; with an output step > 1
// it writes only the (out_step, out_off) grid (zero_phases must be 0: the
// caller zeroes the rest).  tiled_mma_supports: the shape rules, no launch.
cudaError_t launch_tiled_mma(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);
bool tiled_mma_supports(const TiledConv &p, dwconv_dtype dt);
// The same kernel with the fused forward pass (p.fz) compiled in.
cudaError_t launch_tiled_mma_fused(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);
// Tensor-core Toeplitz kernel for large 16-bit filters (tiled_mma_large.cu).
cudaError_t launch_tiled_mma_large(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);

// Stride-2, dilation-1 passes of square 3x3 / 5x5 / 7x7 filters, fp32 / fp16 /
// bf16 (tiled_strided.cu); cudaErrorNotSupported for any other shape.  The
// caller checks the layout (whole 16-byte channel rows, 16-byte aligned
// tensors).  strided_wgrad_slices: the workspace plan (slices of the
// accumulation axis for the workspace bound, 0 if not covered).
cudaError_t launch_strided_fwd(const Shape &s, dwconv_dtype dt, const void *x, const void *w, const float *bias,
                               void *y, const Fuse &fz, cudaStream_t st);
cudaError_t launch_strided_dgrad(const Shape &s, dwconv_dtype dt, const void *dy, const void *w, void *dx,
                                 cudaStream_t st);
int strided_wgrad_slices(const Shape &s, dwconv_dtype dt);
cudaError_t launch_strided_wgrad(const Shape &s, dwconv_dtype dt, const void *x, const void *dy, float *part,
                                 float *dw, cudaStream_t st);

// Whole-map kernels for 7x7 maps, 3x3 / 5x5 / 7x7 filters with "same"
// padding, unit stride, fp32 / fp16 / bf16 (tiled_smallmap.cu): forward and
// stride-1 input gradient (p.flip), and the weight gradient (partials into
// part[Z][FH*FW][C], then the fixed-order reduction into p.out);
// smallmap_wgrad_slices: Z for the workspace bound (0 if not covered).
cudaError_t launch_smallmap(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);
int smallmap_wgrad_slices(const TiledConv &p, dwconv_dtype dt);
cudaError_t launch_smallmap_wgrad(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st);

// Large filters (FW >= 8, any FH), forward and stride-1 input gradient.
cudaError_t launch_tiled_large(const TiledConv &p, dwconv_dtype dt, cudaStream_t st);

// Weight gradient on the tiled path: slices of the accumulation axis for this
// shape (0 if no tiled instance covers it; depends on the shape only), and the
// launch (partials into part[Zc][FH*FW][C], then the fixed-order reduction
// into p.out).
int tiled_wgrad_slices(const TiledConv &p, dwconv_dtype dt);
cudaError_t launch_tiled_wgrad(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st);
// Weight gradient for the filters tiled_wgrad does not compile (large and
// strip filters; p.transpose accepted), tiled_wgrad_large.cu: same contract.
int tiled_wgrad_large_slices(const TiledConv &p, dwconv_dtype dt);
cudaError_t launch_tiled_wgrad_large(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st);
// Tensor-core weight gradient for large 16-bit filters (tiled_mma_wgrad.cu):
// same contract, taken before the CUDA-core kernel when an instance covers it.
int tiled_mma_wgrad_slices(const TiledConv &p, dwconv_dtype dt);
cudaError_t launch_tiled_mma_wgrad(const TiledConv &p, dwconv_dtype dt, float *part, cudaStream_t st);

}  // namespace dwc
