// Host side of the TMA helpers: tensor-map encoding through the driver entry
// point (no link against libcuda), and the device error word.
#include <cudaTypedefs.h>

#include <mutex>

#include "tma.cuh"

namespace dwc {

namespace {

__device__ unsigned g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_err_addr[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

unsigned long long g_err_ctx[kMaxDevices];  // context id the cached address belongs to

}  // namespace

unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return 0;
    if (!ctx) {  // no context in this thread yet: bind the device's primary context
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return 0;
        if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    }
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

unsigned *device_error_word() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const unsigned long long ctx = current_context_id();
    if (!ctx) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_addr[dev] || g_err_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_addr[dev] = static_cast<unsigned *>(p);
        g_err_ctx[dev] = ctx;
    }
    return g_err_addr[dev];
}

cudaError_t take_device_error(cudaStream_t st, unsigned *value) {
    *value = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    unsigned zero = 0;
    e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    if (*value) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));
    return e;
}

bool encode_tmap_4d(CUtensorMap *map, dwconv_dtype dt, const void *base, const uint64_t dims[4],
                    const uint64_t strides[3], const uint32_t box[4], int swizzle, int l2_promotion) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    // The encoder is a driver-API call and needs a context current in the
    // calling thread.  A thread whose first CUDA call is into this library
    // (e.g. a framework's backward-pass worker thread) may have none yet:
    // bind the current device's primary context once per thread, or every
    // tiled kernel would refuse the call and the direct kernel would run.
    thread_local bool context_bound = false;
    if (!context_bound) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
        context_bound = true;
    }
    CUtensorMapDataType t;
    switch (dt) {
        case DWCONV_FP32: t = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; break;
        case DWCONV_FP16: t = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; break;
        case DWCONV_BF16: t = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; break;
        case DWCONV_FP8_E4M3: t = CU_TENSOR_MAP_DATA_TYPE_UINT8; break;  // bytes, moved as they are
        default: return false;
    }
    for (int i = 0; i < 3; ++i)
        if (strides[i] % 16 != 0 || strides[i] >= (1ull << 40)) return false;
    for (int i = 0; i < 4; ++i)
        if (box[i] < 1 || box[i] > 256 || dims[i] < 1 || dims[i] > 0xFFFFFFFFull) return false;
    const cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
    const cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
    const cuuint32_t bd[4] = {box[0], box[1], box[2], box[3]};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    CUtensorMapSwizzle swz;
    switch (swizzle) {
        case 0: swz = CU_TENSOR_MAP_SWIZZLE_NONE; break;
        case 32: swz = CU_TENSOR_MAP_SWIZZLE_32B; break;
        case 64: swz = CU_TENSOR_MAP_SWIZZLE_64B; break;
        default: return false;
    }
    const unsigned esz = dt == DWCONV_FP32 ? 4u : dt == DWCONV_FP8_E4M3 ? 1u : 2u;
    if (swizzle && box[0] * esz != (unsigned)swizzle) return false;
    CUtensorMapL2promotion promo;
    switch (l2_promotion) {
        case 0: promo = CU_TENSOR_MAP_L2_PROMOTION_NONE; break;
        case 64: promo = CU_TENSOR_MAP_L2_PROMOTION_L2_64B; break;
        case 128: promo = CU_TENSOR_MAP_L2_PROMOTION_L2_128B; break;
        case 256: promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B; break;
        default: return false;
    }
    CUresult r = fn(map, t, 4, const_cast<void *>(base), gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swz,
                    promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace dwc
