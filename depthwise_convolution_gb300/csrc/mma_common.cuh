// Pieces shared by the tensor-core (mma.sync) kernels: ldmatrix / stmatrix
// wrappers, the m16n8k16 MMA with fp32 accumulation for fp16 and bf16, and
// the work-unit geometry.
#pragma once

#include "tiled_common.cuh"

namespace dwc {
namespace mma {

using tiled::Unit;

struct GeoM {
    int tiles_h, tiles_w, groups, per_ctile, units;  // groups: image groups (images per unit apart)
};

__device__ __forceinline__ void ldsm_x4_trans(unsigned &r0, unsigned &r1, unsigned &r2, unsigned &r3,
                                              unsigned addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4(unsigned &r0, unsigned &r1, unsigned &r2, unsigned &r3,
                                        unsigned addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(unsigned &r0, unsigned &r1, unsigned addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}
__device__ __forceinline__ void stsm_x4(unsigned addr, unsigned r0, unsigned r1, unsigned r2, unsigned r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(r0),
                 "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

// D (16x8 fp32) += A (16x16) * B (16x8), 16-bit inputs; and packing helpers.
template <typename T> struct MmaOp;
template <> struct MmaOp<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                               unsigned b0, unsigned b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ unsigned pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<unsigned *>(&v);
    }
    static __device__ __forceinline__ unsigned pack_raw(__nv_bfloat16 lo, __nv_bfloat16 hi) {
        return (unsigned)__bfloat16_as_ushort(lo) | ((unsigned)__bfloat16_as_ushort(hi) << 16);
    }
    static __device__ __forceinline__ unsigned short bits(float v) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
};
template <> struct MmaOp<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                               unsigned b0, unsigned b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ unsigned pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<unsigned *>(&v);
    }
    static __device__ __forceinline__ unsigned pack_raw(__half lo, __half hi) {
        return (unsigned)__half_as_ushort(lo) | ((unsigned)__half_as_ushort(hi) << 16);
    }
    static __device__ __forceinline__ unsigned short bits(float v) { return __half_as_ushort(__float2half_rn(v)); }
};

// Unit index -> (channel tile, image, column tile, row band), band fastest.
__device__ __forceinline__ Unit decode(const GeoM &g, int u) {
    Unit r;
    r.ctile = u / g.per_ctile;
    int v = u - r.ctile * g.per_ctile;
    r.band = v % g.tiles_h;
    v /= g.tiles_h;
    r.twi = v % g.tiles_w;
    r.group = v / g.tiles_w;
    return r;
}

// Moves a unit cursor to the next unit (same order as decode); `groups` is
// the number of image groups.
__device__ __forceinline__ void advance(const GeoM &g, int groups, Unit &c) {
    if (++c.band == g.tiles_h) {
        c.band = 0;
        if (++c.twi == g.tiles_w) {
            c.twi = 0;
            if (++c.group == groups) {
                c.group = 0;
                ++c.ctile;
            }
        }
    }
}

// Smallest channel stride (in 16-bit elements) >= n that is 8 mod 16, so the
// 8 channel rows of a stmatrix land in distinct 16-byte bank groups.
constexpr int channel_stride(int n) { return n % 16 == 8 ? n : n + ((8 - n % 16 + 16) % 16); }

constexpr unsigned align1k(unsigned b) { return (b + 1023u) & ~1023u; }

// Tensor map of the kernel's output grid: positions (out_off_h + out_step_h i,
// out_off_w + out_step_w j) of the [N][OHf][OWf][C] tensor p.out, i < OHs,
// j < OWs (the steps folded into the strides, the offsets into the base).
inline bool make_out_map(CUtensorMap *m, const TiledConv &p, dwconv_dtype dt, size_t es, const uint32_t box[4],
                         int swizzle) {
    const char *base = static_cast<const char *>(p.out) + ((size_t)p.out_off_h * p.OWf + p.out_off_w) * p.C * es;
    const uint64_t dims[4] = {(uint64_t)p.C, (uint64_t)p.OWs, (uint64_t)p.OHs, (uint64_t)p.N};
    const uint64_t col = (uint64_t)p.out_step_w * p.C * es, row = (uint64_t)p.out_step_h * p.OWf * p.C * es;
    const uint64_t str[3] = {p.transpose ? row : col, p.transpose ? col : row, (uint64_t)p.OHf * p.OWf * p.C * es};
    return encode_tmap_4d(m, dt, base, dims, str, box, swizzle);
}

}  // namespace mma
}  // namespace dwc
