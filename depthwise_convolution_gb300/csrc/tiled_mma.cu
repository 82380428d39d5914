// Tensor-core forward pass and stride-1 input gradient for 16-bit data and
// 3x3, 5x5 and 7x7 filters: shape rules and the launcher of the plain passes.
// The kernel (Flash-DWC §4.2 Toeplitz packing on mma.sync) is in
// tiled_mma_kernel.cuh, its warp-specialised form for maps wider than 32
// columns in tiled_mma_ring_kernel.cuh; the fused forward pass has its own
// instances in tiled_mma_fused.cu.
#include "tiled_mma_ring_kernel.cuh"

namespace dwc {

bool tiled_mma_supports(const TiledConv &p, dwconv_dtype dt) {
    if (!DWCONV_MMA || p.zero_phases || (dt != DWCONV_FP16 && dt != DWCONV_BF16)) return false;
    if (!((p.FH == 7 && p.FW == 7) || (p.FH == 5 && p.FW == 5) || (p.FH == 3 && p.FW == 3))) return false;
    if (p.OWs <= 8) return false;
    const long long per = (long long)((p.N + 1) / 2) * ((p.OWs + 63) / 8) * p.OHs;  // generous bound
    return per * ((p.C + kCh - 1) / kCh) < (1LL << 30);
}

cudaError_t launch_tiled_mma(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    // Output positions off the (out_step, out_off) grid are not written: a
    // caller with out_step > 1 zeroes them itself.
    if (!DWCONV_MMA || p.zero_phases) return cudaErrorNotSupported;
    if (p.fz.pre() || p.fz.post()) return launch_tiled_mma_fused(p, dt, st);
    switch (dt) {
        case DWCONV_FP16: return by_filter_plain<__half>(p, dt, st);
        case DWCONV_BF16: return by_filter_plain<__nv_bfloat16>(p, dt, st);
        case DWCONV_FP8_E4M3: return p.flip ? cudaErrorNotSupported : by_filter<__nv_fp8_e4m3, false>(p, dt, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
