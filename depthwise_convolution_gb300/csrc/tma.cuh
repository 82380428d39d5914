// TMA (cp.async.bulk.tensor) loads completed on shared-memory mbarriers, with
// bounded waits.
//
// One elected thread issues a whole tile with a single tensor copy; the
// hardware generates zeros for every element outside the tensor, which is how
// the kernels get their padding without fetching it.  Waits spin on
// mbarrier.try_wait at most kSpinLimit times; a wait that runs out sets the
// library's device error word (read by dwconv_check_device_errors) and the
// kernel returns instead of hanging.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace dwc {

constexpr unsigned kSpinLimit = 1u << 26;  // try_wait polls before giving up (seconds)

// Unique id of the context current in the calling thread (the device's
// primary context, made current if none is), 0 if it cannot be read.  A
// device reset destroys the context and the next one gets a new id, so caches
// of device addresses keyed by it never hand out an address of a context that
// no longer exists.
unsigned long long current_context_id();

// Device error word: bit 0 = a bounded wait gave up.  Its address is looked up
// once per context.
unsigned *device_error_word();
// Reads and clears the error word of the current device (after syncing `st`).
cudaError_t take_device_error(cudaStream_t st, unsigned *value);

// 4-D tiled tensor map, dims innermost first (C, W, H, N), strides in bytes
// for dims 1..3, box in elements; swizzle: shared-memory swizzle span in
// bytes (0 = none, 32 or 64; the inner box row must then be exactly that
// long); l2_promotion: L2 fetch size in bytes (0, 64, 128 or 256).  Returns
// false if the driver rejects it.
//
// 64 is the default: a unit's box row is one 32-channel slice (64 bytes for
// 16-bit data) of a pixel, and with 128-byte promotion the halo rows that
// vertically adjacent units share were fetched from DRAM again (measured:
// 1.8x the unique input bytes read, against 1.04x with 64-byte promotion).
#ifndef DWCONV_L2_PROMO
#define DWCONV_L2_PROMO 64
#endif
bool encode_tmap_4d(CUtensorMap *map, dwconv_dtype dt, const void *base, const uint64_t dims[4],
                    const uint64_t strides[3], const uint32_t box[4], int swizzle = 0,
                    int l2_promotion = DWCONV_L2_PROMO);

__device__ __forceinline__ unsigned smem_addr(const void *p) {
    return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Plain arrival (count 1) on a barrier, e.g. a consumer releasing a slot.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
        : "memory");
}

// Waits for the barrier phase with the given parity; false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity) {
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
    }
    return false;
}

__device__ __forceinline__ void report_timeout(unsigned *err) {
    if (err) atomicOr(err, 1u);
}

}  // namespace dwc
