// dwconv_bwd_filter_static: the weight gradient for callers that cannot
// allocate device memory.
//
// dwconv_bwd_filter needs a scratch buffer for the partial sums of its split
// reduction, and leaves it to the caller to provide one.  Some callers have no
// way to get one: code that runs under a host framework whose caching
// allocator already owns the device memory (a plugin or custom operator that
// must not call cudaMalloc behind the framework's back, and may not be handed
// a buffer either), or deployments that fix their memory plan at start-up and
// forbid any allocation afterwards.  This entry point serves them: its scratch
// is a fixed-size array in the library's own device image, so the call itself
// allocates nothing.
//
// The array is a file-scope __device__ variable.  Host code cannot use its
// name as a device address (on the host the name denotes a host-side shadow
// object), so the first call on each device asks the runtime for the array's
// device address with cudaGetSymbolAddress, with that device current, and
// caches it; later calls on that device reuse the cached address.  The cache
// remembers which context the address belongs to: after a device reset the
// module is loaded again into a new context, possibly elsewhere, and the next
// call looks the address up again.
#include <mutex>

#include "common.cuh"
#include "tma.cuh"

namespace {

// Held by every GPU that loads this library until the process exits.
static __device__ __align__(256) unsigned char g_scratch[DWCONV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];            // device address of g_scratch, per device
unsigned long long g_scratch_ctx[kMaxDevices];  // the context that address belongs to

// Device address of g_scratch on the current device, looked up once per
// device and context.
cudaError_t scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const unsigned long long ctx = dwc::current_context_id();
    if (!ctx) return cudaErrorInvalidValue;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" dwconv_status dwconv_bwd_filter_static(int N, int H, int W, int C, int FH, int FW,
                                                  int stride, int dilation, int pad,
                                                  dwconv_dtype dtype, const void *x,
                                                  const void *dy, float *dw,
                                                  dwconv_stream stream) {
    const size_t need = dwconv_bwd_filter_workspace_size(N, H, W, C, FH, FW, stride, dilation,
                                                         pad, dtype);
    if (need == 0)  // invalid arguments: let the regular entry point name the error
        return dwconv_bwd_filter(N, H, W, C, FH, FW, stride, dilation, pad, dtype, x, dy, dw,
                                 nullptr, 0, stream);
    if (need > DWCONV_STATIC_SCRATCH_BYTES) return DWCONV_ERR_INVALID_ARG;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return DWCONV_ERR_CUDA;
    // Every partial sum the reduction reads is written earlier in the same
    // call, so leftovers from a previous call need no clearing.
    return dwconv_bwd_filter(N, H, W, C, FH, FW, stride, dilation, pad, dtype, x, dy, dw, scratch,
                             DWCONV_STATIC_SCRATCH_BYTES, stream);
}
