// Pipe-rate probes: the measured denominators beside the roofline of the
// CUDA-core kernels (FP32 and mixed-precision FMA), and the rates of the two
// tensor-core instruction families the convolution kernels could use (warp
// mma.sync, and tcgen05.mma from shared-memory descriptors with the
// accumulator in tensor memory).  Built as libdwprobe.so, separate from the
// convolution library; bench.py and the profile summaries call it.
//
// Every kernel runs independent chains for a few milliseconds on one CTA per
// SM (grid = SM count); operands are constants (only the rate is measured).
// The tcgen05 kernel allocates 256 tensor-memory columns per CTA, waits on its
// commit barrier a bounded number of polls (setting an error word instead of
// hanging), and frees the columns on every path.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ unsigned g_probe_err;

template <int KIND, int CH>
__global__ void fma_kernel(float *out, int iters) {
    // KIND 0: fp32 FFMA; 1: packed fma.rn.f32x2; 2: fma.rn.f32.f16; 3: fma.rn.f32.bf16.
    float acc[CH][2];
#pragma unroll
    for (int i = 0; i < CH; ++i) acc[i][0] = acc[i][1] = threadIdx.x * 1e-3f + i;
    const float a = 1.0001f, b = 1e-6f;
    const unsigned short h = (KIND == 3 ? 0x3f80 : 0x3c00) ^ (threadIdx.x & 1);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            if constexpr (KIND == 0) {
                acc[i][0] = fmaf(acc[i][0], a, b);
            } else if constexpr (KIND == 1) {
                float2 v = make_float2(acc[i][0], acc[i][1]);
                v = __ffma2_rn(v, make_float2(a, a), make_float2(b, b));
                acc[i][0] = v.x;
                acc[i][1] = v.y;
            } else if constexpr (KIND == 2) {
                asm volatile("fma.rn.f32.f16 %0, %1, %1, %0;" : "+f"(acc[i][0]) : "h"(h));
            } else {
                asm volatile("fma.rn.f32.bf16 %0, %1, %1, %0;" : "+f"(acc[i][0]) : "h"(h));
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < CH; ++i) s += acc[i][0] + acc[i][1];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

template <int CH>
__global__ void mma_sync_kernel(float *out, int iters) {
    const unsigned a0 = 0x3f803f80u ^ threadIdx.x, b0 = 0x3c003c00u;
    float d[CH][4];
#pragma unroll
    for (int c = 0; c < CH; ++c) d[c][0] = d[c][1] = d[c][2] = d[c][3] = 0.f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < CH; ++c)
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
                : "r"(a0), "r"(a0), "r"(a0), "r"(a0), "r"(b0), "r"(b0));
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) s += d[c][0] + d[c][1] + d[c][2] + d[c][3];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__device__ __forceinline__ unsigned saddr(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor (no swizzle): start >> 4 at bits 0-13,
// leading-dimension byte offset >> 4 at 16-29, stride byte offset >> 4 at
// 32-45, descriptor version 1 at bits 46-47.
__device__ __forceinline__ uint64_t smem_desc(unsigned addr, unsigned lbo, unsigned sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// (bits 7-9 = 1) and B (bits 10-12 = 1), both K-major, N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
__device__ __forceinline__ unsigned instr_desc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((unsigned)(N >> 3) << 17) | ((unsigned)(M >> 4) << 24);
}

constexpr int kAB = 128 * 16 * 2, kBB = 256 * 16 * 2, kCols = 256;
constexpr unsigned kPolls = 1u << 26;

__device__ bool wait_parity(uint64_t *bar, unsigned phase) {
    for (unsigned s = 0; s < kPolls; ++s) {
        unsigned d;
        asm volatile(
            "{ .reg .pred q; mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2; selp.u32 %0, 1, 0, q; }"
            : "=r"(d)
            : "r"(saddr(bar)), "r"(phase)
            : "memory");
        if (d) return true;
    }
    return false;
}

// One CTA per SM, 128 threads; warps 0..nw-1 each issue (from one lane) `per`
// MMAs of M x N x 16 into nd accumulators of their own, commit, wait, repeat.
__global__ void tcgen05_kernel(int M, int N, int iters, int per, int nd, int nw) {
    __shared__ __align__(1024) unsigned char A[kAB];
    __shared__ __align__(1024) unsigned char B[kBB];
    __shared__ __align__(8) uint64_t bars[4];
    __shared__ unsigned tmem_base;
    const int tid = threadIdx.x, warp = tid / 32;
    for (int i = tid; i < kAB / 4; i += blockDim.x) reinterpret_cast<unsigned *>(A)[i] = 0;
    for (int i = tid; i < kBB / 4; i += blockDim.x) reinterpret_cast<unsigned *>(B)[i] = 0;
    if (tid == 0) {
        for (int w = 0; w < 4; ++w) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&bars[w])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tmem_base)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the zero operands, visible to the tensor core
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const unsigned taddr = tmem_base;
    if (tid % 32 == 0 && warp < nw) {
        uint64_t *bar = &bars[warp];
        const unsigned dbase = taddr + (unsigned)(warp * nd * N);
        // K-major, no swizzle: core matrix = 8 rows x 16 bytes; K direction 128 B apart, M/N 256 B.
        const uint64_t ad = smem_desc(saddr(A), 128, 256), bd = smem_desc(saddr(B), 128, 256);
        const unsigned id = instr_desc(M, N);
        unsigned phase = 0;
        for (int it = 0; it < iters; ++it) {
            for (int j = 0; j < per; ++j) {
                const unsigned accum = it ? 1u : 0u;
                const unsigned d = dbase + (unsigned)((j % nd) * N);
                asm volatile(
                    "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
                    " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
                    "l"(ad), "l"(bd), "r"(id), "r"(accum)
                    : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             saddr(bar))
                         : "memory");
            if (!wait_parity(bar, phase)) {
                atomicOr(&g_probe_err, 1u);
                wait_parity(bar, phase);  // give the MMAs in flight a second bounded chance
                break;
            }
            phase ^= 1;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kCols) : "memory");
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

// Mean milliseconds of `reps` launches after one untimed launch.
template <typename F>
cudaError_t time_ms(F launch, int reps, float *ms) {
    cudaEvent_t e0, e1;
    cudaError_t e = cudaEventCreate(&e0);
    if (e != cudaSuccess) return e;
    e = cudaEventCreate(&e1);
    if (e != cudaSuccess) return e;
    launch();
    cudaEventRecord(e0);
    for (int r = 0; r < reps; ++r) launch();
    cudaEventRecord(e1);
    e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
    *ms /= reps;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return e;
}

}  // namespace

extern "C" {

// FMA pipe rate in TFLOP/s (2 flops per fused multiply-add; 4 for the packed
// pair): kind 0 fp32 FFMA, 1 packed fma.rn.f32x2, 2 fma.rn.f32.f16, 3
// fma.rn.f32.bf16; `warps` warps per SM, 8 independent chains per thread.
int dwp_fma_rate(int kind, int warps, int iters, double *tflops) {
    const int sms = sm_count(), block = 32 * warps;
    if (sms <= 0 || warps < 1 || warps > 32 || iters < 1 || kind < 0 || kind > 3) return -1;
    float *out = nullptr;
    cudaError_t e = cudaMalloc(&out, (size_t)sms * block * sizeof(float));
    if (e != cudaSuccess) return (int)e;
    float ms = 0.f;
    auto go = [&](auto k) { return time_ms([&] { k<<<sms, block>>>(out, iters); }, 5, &ms); };
    switch (kind) {
        case 0: e = go(fma_kernel<0, 8>); break;
        case 1: e = go(fma_kernel<1, 8>); break;
        case 2: e = go(fma_kernel<2, 8>); break;
        default: e = go(fma_kernel<3, 8>); break;
    }
    cudaFree(out);
    if (e != cudaSuccess) return (int)e;
    const double per_fma = kind == 1 ? 4.0 : 2.0;
    *tflops = per_fma * 8.0 * iters * (double)block * sms / (ms * 1e-3) / 1e12;
    return 0;
}

// Warp-level mma.sync m16n8k16 bf16 -> fp32 rate in TFLOP/s, `warps` warps per
// SM, 8 independent accumulators per warp.
int dwp_mma_sync_rate(int warps, int iters, double *tflops) {
    const int sms = sm_count(), block = 32 * warps;
    if (sms <= 0 || warps < 1 || warps > 32 || iters < 1) return -1;
    float *out = nullptr;
    cudaError_t e = cudaMalloc(&out, (size_t)sms * block * sizeof(float));
    if (e != cudaSuccess) return (int)e;
    float ms = 0.f;
    e = time_ms([&] { mma_sync_kernel<8><<<sms, block>>>(out, iters); }, 5, &ms);
    cudaFree(out);
    if (e != cudaSuccess) return (int)e;
    *tflops = 2.0 * 16 * 8 * 16 * 8.0 * iters * (double)warps * sms / (ms * 1e-3) / 1e12;
    return 0;
}

// tcgen05.mma kind::f16 (bf16 operands from shared memory, fp32 accumulator in
// tensor memory) rate in TFLOP/s for an M x N x 16 shape: nw issuing warps
// per SM, each with nd accumulators and `per` MMAs between commits.
// *timeouts: nonzero if a bounded wait gave up (the rate is then invalid).
int dwp_tcgen05_rate(int M, int N, int per, int nd, int nw, int iters, double *tflops, unsigned *timeouts) {
    const int sms = sm_count();
    if (sms <= 0 || !(M == 64 || M == 128) || N < 8 || N > 256 || N % (M == 64 ? 8 : 16) != 0 || nd < 1 ||
        nw < 1 || nw > 4 || per < 1 || iters < 1 || nd * N * nw > kCols)
        return -1;
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyToSymbol(g_probe_err, &zero, sizeof(zero));
    if (e != cudaSuccess) return (int)e;
    float ms = 0.f;
    e = time_ms([&] { tcgen05_kernel<<<sms, 128>>>(M, N, iters, per, nd, nw); }, 3, &ms);
    if (e != cudaSuccess) return (int)e;
    e = cudaMemcpyFromSymbol(timeouts, g_probe_err, sizeof(unsigned));
    if (e != cudaSuccess) return (int)e;
    *tflops = 2.0 * M * N * 16 * (double)per * iters * nw * sms / (ms * 1e-3) / 1e12;
    return 0;
}

}  // extern "C"
