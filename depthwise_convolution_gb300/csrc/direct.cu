// Direct kernels: one thread per output element, any shape and stride.
//
// These cover every request the register-tiled kernels do not (odd channel
// counts such as the 5-channel int8 case, strides and dilations without a
// tiled instance) and are the simplest statement of each pass on the GPU.
// Padding is generated: a tap outside the input contributes nothing.
#include "common.cuh"

namespace dwc {
namespace {

constexpr int kThreads = 256;

int grid_for(long long total) {
    long long blocks = (total + kThreads - 1) / kThreads;
    long long cap = (long long)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

// Forward, floating point: fp32 accumulation, bias first, taps fh-major;
// optional BN+Act prologue on every input value read (rounded back to T, as
// the unfused layer stores it) and affine+activation epilogue.
template <typename T>
__global__ void __launch_bounds__(kThreads) fwd_direct_fp(Shape s, const T *__restrict__ x,
                                                          const T *__restrict__ w,
                                                          const float *__restrict__ bias,
                                                          typename OutOf<T>::type *__restrict__ y, long long total,
                                                          Fuse fz) {
    const bool pre = fz.pre(), post = fz.post();
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        int c = (int)(idx % s.C);
        long long t = idx / s.C;
        int ow = (int)(t % s.OW);
        t /= s.OW;
        int oh = (int)(t % s.OH);
        long long n = t / s.OH;
        float acc = bias ? bias[c] : 0.f;
        const Affine ain = pre ? affine_in(fz, c) : Affine{1.f, 0.f};
        for (int fh = 0; fh < s.FH; ++fh) {
            int ih = oh * s.SH - s.PH + fh * s.DH;
            if (ih < 0 || ih >= s.H) continue;
            const T *xrow = x + ((n * s.H + ih) * s.W) * (long long)s.C + c;
            const T *wrow = w + (long long)fh * s.FW * s.C + c;
            for (int fw = 0; fw < s.FW; ++fw) {
                int iw = ow * s.SW - s.PW + fw * s.DW;
                if (iw < 0 || iw >= s.W) continue;
                float xv = to_f32(xrow[(long long)iw * s.C]);
                if (pre) xv = to_f32(from_f32<T>(apply(ain, xv, fz.in_act)));
                acc = fmaf(to_f32(wrow[(long long)fw * s.C]), xv, acc);
            }
        }
        if (post) acc = apply(affine_out(fz, c), acc, fz.out_act);
        y[idx] = from_f32<typename OutOf<T>::type>(acc);
    }
}

// Forward, int8 x int8 -> int32.  Products are exact in int32; the running
// sum is kept in uint32 so that overflow wraps (two's complement) instead of
// being undefined.
__global__ void __launch_bounds__(kThreads) fwd_direct_i8(Shape s, const int8_t *__restrict__ x,
                                                          const int8_t *__restrict__ w,
                                                          const int32_t *__restrict__ bias,
                                                          int32_t *__restrict__ y,
                                                          long long total) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        int c = (int)(idx % s.C);
        long long t = idx / s.C;
        int ow = (int)(t % s.OW);
        t /= s.OW;
        int oh = (int)(t % s.OH);
        long long n = t / s.OH;
        uint32_t acc = bias ? (uint32_t)bias[c] : 0u;
        for (int fh = 0; fh < s.FH; ++fh) {
            int ih = oh * s.SH - s.PH + fh * s.DH;
            if (ih < 0 || ih >= s.H) continue;
            for (int fw = 0; fw < s.FW; ++fw) {
                int iw = ow * s.SW - s.PW + fw * s.DW;
                if (iw < 0 || iw >= s.W) continue;
                int prod = (int)w[((long long)fh * s.FW + fw) * s.C + c] *
                           (int)x[((n * s.H + ih) * s.W + iw) * (long long)s.C + c];
                acc += (uint32_t)prod;
            }
        }
        y[idx] = (int32_t)acc;
    }
}

// Input gradient in gather form: dx[ih] sums the taps fh whose output row
// oh = (ih + P - fh*D)/S is a whole number inside [0, OH); likewise along w.
template <typename T>
__global__ void __launch_bounds__(kThreads) dgrad_direct(Shape s, const T *__restrict__ dy,
                                                         const T *__restrict__ w,
                                                         T *__restrict__ dx, long long total) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        int c = (int)(idx % s.C);
        long long t = idx / s.C;
        int iw = (int)(t % s.W);
        t /= s.W;
        int ih = (int)(t % s.H);
        long long n = t / s.H;
        float acc = 0.f;
        for (int fh = 0; fh < s.FH; ++fh) {
            int th = ih + s.PH - fh * s.DH;
            if (th < 0) break;                  // decreases with fh
            if (th % s.SH != 0) continue;
            int oh = th / s.SH;
            if (oh >= s.OH) continue;
            for (int fw = 0; fw < s.FW; ++fw) {
                int tw = iw + s.PW - fw * s.DW;
                if (tw < 0) break;
                if (tw % s.SW != 0) continue;
                int ow = tw / s.SW;
                if (ow >= s.OW) continue;
                acc = fmaf(to_f32(w[((long long)fh * s.FW + fw) * s.C + c]),
                           to_f32(dy[((n * s.OH + oh) * s.OW + ow) * (long long)s.C + c]), acc);
            }
        }
        dx[idx] = from_f32<T>(acc);
    }
}

// Weight gradient, first pass.  Block (32 channels x 8 position lanes) handles
// one filter tap and one slice z of the N*OH*OW axis; the 8 lanes are summed
// in a fixed order and written to part[z][tap][c].
template <typename T>
__global__ void __launch_bounds__(kThreads) wgrad_direct(Shape s, const T *__restrict__ x,
                                                         const T *__restrict__ dy,
                                                         float *__restrict__ part, int Z) {
    __shared__ float red[8][33];
    const int c = blockIdx.x * 32 + threadIdx.x;
    const int tap = blockIdx.y;
    const int fh = tap / s.FW, fw = tap % s.FW;
    const int z = blockIdx.z;
    const long long positions = (long long)s.N * s.OH * s.OW;
    const long long p0 = positions * z / Z, p1 = positions * (z + 1) / Z;
    float acc = 0.f;
    if (c < s.C) {
        for (long long p = p0 + threadIdx.y; p < p1; p += 8) {
            int ow = (int)(p % s.OW);
            long long t = p / s.OW;
            int oh = (int)(t % s.OH);
            long long n = t / s.OH;
            int ih = oh * s.SH - s.PH + fh * s.DH;
            int iw = ow * s.SW - s.PW + fw * s.DW;
            if (ih < 0 || ih >= s.H || iw < 0 || iw >= s.W) continue;
            acc = fmaf(to_f32(dy[p * s.C + c]),
                       to_f32(x[((n * s.H + ih) * s.W + iw) * (long long)s.C + c]), acc);
        }
    }
    red[threadIdx.y][threadIdx.x] = acc;
    __syncthreads();
    if (threadIdx.y == 0 && c < s.C) {
        float sum = 0.f;
        for (int k = 0; k < 8; ++k) sum += red[k][threadIdx.x];
        part[((long long)z * s.FH * s.FW + tap) * s.C + c] = sum;
    }
}

// dw[i] = sum over slices z of part[z][i], in a fixed order: warp r of a
// block sums the slices z = r, r + 8, r + 16, ... (increasing), then the 8
// warp sums are added in warp order.  A block covers 32 consecutive elements
// (coalesced loads per slice); 8 independent chains per element keep enough
// loads in flight for a grid of count/32 blocks.
constexpr int kReduceWarps = 8;
__global__ void __launch_bounds__(32 * kReduceWarps) wgrad_reduce(const float *__restrict__ part, int Z,
                                                                  long long count, float *__restrict__ dw) {
    __shared__ float acc[kReduceWarps][32];
    const int lane = threadIdx.x % 32, r = threadIdx.x / 32;
    const long long i = blockIdx.x * 32LL + lane;
    // Launched as a programmatic dependent of the kernel that writes `part`:
    // wait here until that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    float sum = 0.f;
    if (i < count) {
        // Loads in batches of 8 (all in flight at once), added in slice order.
        int z = r;
        for (; z + 7 * kReduceWarps < Z; z += 8 * kReduceWarps) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = part[(long long)(z + q * kReduceWarps) * count + i];
#pragma unroll
            for (int q = 0; q < 8; ++q) sum += v[q];
        }
        for (; z < Z; z += kReduceWarps) sum += part[(long long)z * count + i];
    }
    acc[r][lane] = sum;
    __syncthreads();
    if (r == 0 && i < count) {
        float t = acc[0][lane];
        for (int q = 1; q < kReduceWarps; ++q) t += acc[q][lane];
        dw[i] = t;
    }
}

// Bias-gradient slices: block (channel block cb, slice z) sums dy over the
// positions of slice z for channels 32 cb + lane; warp r takes positions
// r, r + 8, ... of the slice (in increasing order) and the 8 warp sums are
// added in warp order, so the result does not depend on scheduling.
template <typename T>
__global__ void __launch_bounds__(256) bias_slice_kernel(const T *__restrict__ dy, long long P, int C, int Z,
                                                        float *__restrict__ part) {
    __shared__ float acc[8][32];
    const int lane = threadIdx.x % 32, r = threadIdx.x / 32;
    const int c = blockIdx.x * 32 + lane;
    const int z = blockIdx.y;
    const long long p0 = P * z / Z, p1 = P * (z + 1) / Z;
    float sum = 0.f;
    if (c < C)
        for (long long q = p0 + r; q < p1; q += 8) sum += to_f32(dy[q * C + c]);
    acc[r][lane] = sum;
    __syncthreads();
    if (r == 0 && c < C) {
        float t = acc[0][lane];
        for (int q = 1; q < 8; ++q) t += acc[q][lane];
        part[(long long)z * C + c] = t;
    }
}

}  // namespace

int bias_slices(long long P, int C, bool launch) {
    const long long cblocks = (C + 31) / 32;
    long long z = (4LL * plan_sms(launch) + cblocks - 1) / cblocks;  // about 4 blocks per SM
    if (z > P) z = P;
    if (z > 4096) z = 4096;
    return (int)(z < 1 ? 1 : z);
}

cudaError_t launch_bias_slices(long long P, int C, dwconv_dtype dt, const void *dy, float *part, int Z,
                               cudaStream_t st) {
    const dim3 grid((unsigned)((C + 31) / 32), (unsigned)Z);
    switch (dt) {
        case DWCONV_FP32: bias_slice_kernel<float><<<grid, 256, 0, st>>>((const float *)dy, P, C, Z, part); break;
        case DWCONV_FP16: bias_slice_kernel<__half><<<grid, 256, 0, st>>>((const __half *)dy, P, C, Z, part); break;
        case DWCONV_BF16:
            bias_slice_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)dy, P, C, Z, part);
            break;
        default: return cudaErrorInvalidValue;
    }
    note_launches(1);
    note_kernel("bias_slices");
    return cudaGetLastError();
}

cudaError_t launch_fwd_direct(const Shape &s, dwconv_dtype dt, const void *x, const void *w,
                              const void *bias, void *y, const Fuse &fz, cudaStream_t st) {
    const long long total = (long long)s.N * s.OH * s.OW * s.C;
    const int grid = grid_for(total);
    switch (dt) {
        case DWCONV_INT8:
            fwd_direct_i8<<<grid, kThreads, 0, st>>>(s, (const int8_t *)x, (const int8_t *)w,
                                                      (const int32_t *)bias, (int32_t *)y, total);
            break;
        case DWCONV_FP32:
            fwd_direct_fp<float><<<grid, kThreads, 0, st>>>(s, (const float *)x, (const float *)w,
                                                            (const float *)bias, (float *)y, total, fz);
            break;
        case DWCONV_FP16:
            fwd_direct_fp<__half><<<grid, kThreads, 0, st>>>(s, (const __half *)x, (const __half *)w,
                                                             (const float *)bias, (__half *)y, total, fz);
            break;
        case DWCONV_BF16:
            fwd_direct_fp<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
                s, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)w, (const float *)bias,
                (__nv_bfloat16 *)y, total, fz);
            break;
        case DWCONV_FP8_E4M3:  // e4m3 x and w, bf16 y
            fwd_direct_fp<__nv_fp8_e4m3><<<grid, kThreads, 0, st>>>(
                s, (const __nv_fp8_e4m3 *)x, (const __nv_fp8_e4m3 *)w, (const float *)bias, (__nv_bfloat16 *)y,
                total, fz);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    note_launches(1);
    note_kernel("direct_fwd");
    return cudaGetLastError();
}

cudaError_t launch_dgrad_direct(const Shape &s, dwconv_dtype dt, const void *dy, const void *w,
                                void *dx, cudaStream_t st) {
    const long long total = (long long)s.N * s.H * s.W * s.C;
    const int grid = grid_for(total);
    switch (dt) {
        case DWCONV_FP32:
            dgrad_direct<float><<<grid, kThreads, 0, st>>>(s, (const float *)dy, (const float *)w,
                                                           (float *)dx, total);
            break;
        case DWCONV_FP16:
            dgrad_direct<__half><<<grid, kThreads, 0, st>>>(s, (const __half *)dy, (const __half *)w,
                                                            (__half *)dx, total);
            break;
        case DWCONV_BF16:
            dgrad_direct<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
                s, (const __nv_bfloat16 *)dy, (const __nv_bfloat16 *)w, (__nv_bfloat16 *)dx, total);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    note_launches(1);
    note_kernel("direct_dgrad");
    return cudaGetLastError();
}

cudaError_t launch_wgrad_direct(const Shape &s, dwconv_dtype dt, const void *x, const void *dy,
                                float *part, int Z, cudaStream_t st) {
    dim3 grid((s.C + 31) / 32, s.FH * s.FW, Z), block(32, 8);
    switch (dt) {
        case DWCONV_FP32:
            wgrad_direct<float><<<grid, block, 0, st>>>(s, (const float *)x, (const float *)dy, part, Z);
            break;
        case DWCONV_FP16:
            wgrad_direct<__half><<<grid, block, 0, st>>>(s, (const __half *)x, (const __half *)dy, part, Z);
            break;
        case DWCONV_BF16:
            wgrad_direct<__nv_bfloat16><<<grid, block, 0, st>>>(
                s, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)dy, part, Z);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    note_launches(1);
    note_kernel("direct_wgrad");
    return cudaGetLastError();
}

cudaError_t launch_wgrad_reduce(const float *part, int Z, long long count, float *dw,
                                cudaStream_t st) {
    const long long blocks = (count + 31) / 32;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    // Programmatic dependent launch: the reduction's blocks are scheduled as
    // the producing kernel drains instead of after a full launch gap; they
    // wait (griddepcontrol.wait) for its completion before reading.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(32 * kReduceWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, wgrad_reduce, part, Z, count, dw);
    note_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dwc
