// Self-test of the library's failure detection, for callers and tests that
// want to see the timeout path work without a fault or a hang.
//
// Every tiled kernel waits for its TMA copies on shared-memory mbarriers with
// a bounded number of polls; a wait that runs out sets the device error word
// and the kernel returns (dwconv_check_device_errors then reports
// DWCONV_ERR_TIMEOUT).  The kernel here makes the same kind of wait on a
// barrier that nothing completes -- no copy is issued and no thread arrives --
// with a short bound, gives up, and records the timeout exactly as the
// production kernels do.  It launches one thread, touches no caller memory and
// leaves the context usable.
#include "dwconv.h"
#include "tma.cuh"

namespace dwc {
namespace {

constexpr unsigned kSelfTestPolls = 1u << 14;  // a few milliseconds at most

__global__ void wait_on_barrier_nothing_completes(unsigned *err) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    mbar_fence_init();
    const unsigned a = smem_addr(&bar);
    unsigned done = 0;
    for (unsigned i = 0; i < kSelfTestPolls && !done; ++i)
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(0u)
            : "memory");
    if (!done) report_timeout(err);
}

}  // namespace
}  // namespace dwc

extern "C" dwconv_status dwconv_selftest_timeout(dwconv_stream stream) {
    unsigned *err = dwc::device_error_word();
    if (!err) return DWCONV_ERR_CUDA;
    dwc::wait_on_barrier_nothing_completes<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
    dwc::note_launches(1);
    return cudaGetLastError() == cudaSuccess ? DWCONV_OK : DWCONV_ERR_CUDA;
}
