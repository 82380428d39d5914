// Instances of the tensor-core kernel (tiled_mma_kernel.cuh) with the fused
// forward pass compiled in (Flash-DWC §5.2 "Kernel fusion"): the BN+Act
// prologue is applied while the staged input is transposed into the
// channel-major operand buffer, the affine+activation epilogue to the fp32
// sums before they are rounded.
#include "tiled_mma_kernel.cuh"

namespace dwc {

cudaError_t launch_tiled_mma_fused(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (!DWCONV_MMA || p.zero_phases || p.flip) return cudaErrorNotSupported;
    switch (dt) {
        case DWCONV_FP16: return by_filter<__half, true>(p, dt, st);
        case DWCONV_BF16: return by_filter<__nv_bfloat16, true>(p, dt, st);
        case DWCONV_FP8_E4M3: return p.flip ? cudaErrorNotSupported : by_filter<__nv_fp8_e4m3, true>(p, dt, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
