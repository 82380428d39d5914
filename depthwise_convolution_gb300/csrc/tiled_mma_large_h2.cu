// Tensor-core large-filter forward pass / stride-1 input gradient: plain
// instances for filter heights 19, 21, 23 and 25 (kernel in tiled_mma_large_kernel.cuh).
// A height runs with the number of 16-input blocks its square filter needs,
// ceil((FH + 7) / 16); a narrower or wider filter of that height runs here
// when it needs the same number.
#include "tiled_mma_large_kernel.cuh"

namespace dwc {
namespace {

template <typename T>
cudaError_t by_height(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    const int nkb = (p.FW + 7 + 15) / 16;
    if (p.FH == 19 && nkb == 2) return large_by_width<T, 19, 2, false>(p, dt, st);
    if (p.FH == 21 && nkb == 2) return large_by_width<T, 21, 2, false>(p, dt, st);
    if (p.FH == 23 && nkb == 2) return large_by_width<T, 23, 2, false>(p, dt, st);
    if (p.FH == 25 && nkb == 2) return large_by_width<T, 25, 2, false>(p, dt, st);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_mma_large_h2(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (p.fz.pre() || p.fz.post()) return cudaErrorNotSupported;
    switch (dt) {
        case DWCONV_FP16: return by_height<__half>(p, dt, st);
        case DWCONV_BF16: return by_height<__nv_bfloat16>(p, dt, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace dwc
