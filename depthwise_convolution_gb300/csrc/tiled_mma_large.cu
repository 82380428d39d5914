// Tensor-core forward pass and stride-1 input gradient for large 16-bit
// filters: shape rules and the launcher.  The kernel (Flash-DWC §4.2 Toeplitz
// packing on mma.sync) is in tiled_mma_large_kernel.cuh; this file holds the
// 13- and 31-row instances (plain and fused) and the 5-row strip instance, the
// tiled_mma_large_h*.cu files the other odd heights from 9 to 29 (plain).
#include "tiled_mma_large_kernel.cuh"

namespace dwc {
namespace {

// Filter blocks for a width: the band of 8 outputs spans 8 + FW - 1 inputs.
template <typename T, bool FUSE>
cudaError_t large_by_filter(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    const int nkb = (p.FW + 7 + 15) / 16;
    if (p.FH == 31 && nkb == 3) return large_by_width<T, 31, 3, FUSE>(p, dt, st);
    if (p.FH == 13 && nkb == 2) return large_by_width<T, 13, 2, FUSE>(p, dt, st);
    if (p.FH == 5 && nkb == 4) return large_by_width<T, 5, 4, FUSE>(p, dt, st);  // 5 x 51 strips (either way)
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t large_dispatch(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (p.fz.pre() || p.fz.post()) return p.flip ? cudaErrorNotSupported : large_by_filter<T, true>(p, dt, st);
    cudaError_t e = large_by_filter<T, false>(p, dt, st);
    if (e == cudaErrorNotSupported) e = launch_mma_large_h1(p, dt, st);
    if (e == cudaErrorNotSupported) e = launch_mma_large_h2(p, dt, st);
    if (e == cudaErrorNotSupported) e = launch_mma_large_h3(p, dt, st);
    return e;
}

}  // namespace

#ifndef DWCONV_MMA_LARGE
#define DWCONV_MMA_LARGE 1  // 0: leave large filters to the CUDA-core kernel
#endif

cudaError_t launch_tiled_mma_large(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (!DWCONV_MMA_LARGE || p.zero_phases || p.out_step_h != 1 || p.out_step_w != 1) return cudaErrorNotSupported;
    switch (dt) {
        case DWCONV_FP16: return large_dispatch<__half>(p, dt, st);
        case DWCONV_BF16: return large_dispatch<__nv_bfloat16>(p, dt, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
