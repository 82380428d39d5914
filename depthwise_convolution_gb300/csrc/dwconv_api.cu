// C ABI of libdwconv: argument validation, shape math, kernel selection.
//
// Every entry point validates all arguments on the host before it touches
// the CUDA runtime, so a rejected call enqueues nothing (and needs no GPU).
#include <algorithm>
#include <atomic>
#include <climits>
#include <mutex>
#include <unordered_map>

#include <utility>

#include "common.cuh"
#include "tma.cuh"

namespace dwc {

namespace {
std::atomic<unsigned long long> g_launches{0};
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_per_sm[kMaxDevices];
}  // namespace

void note_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {
thread_local const char *t_last_kernel = "none";
}
void note_kernel(const char *family) { t_last_kernel = family; }

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        g_sm_count[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

namespace {
struct SetupKey {
    const void *kern;
    unsigned long long ctx;
    int threads;
    size_t smem;
    bool operator==(const SetupKey &o) const {
        return kern == o.kern && ctx == o.ctx && threads == o.threads && smem == o.smem;
    }
};
struct SetupHash {
    size_t operator()(const SetupKey &k) const {
        size_t h = std::hash<const void *>()(k.kern);
        h = h * 1000003u ^ std::hash<unsigned long long>()(k.ctx);
        h = h * 1000003u ^ (size_t)k.threads;
        return h * 1000003u ^ k.smem;
    }
};
std::mutex g_setup_mu;
std::unordered_map<SetupKey, int, SetupHash> g_occupancy;    // (kernel, context, threads, smem) -> CTAs per SM
std::unordered_map<SetupKey, size_t, SetupHash> g_smem_limit;  // (kernel, context) -> largest limit set
}  // namespace

cudaError_t kernel_setup(const void *kern, int threads, size_t smem, int *per_sm) {
    const unsigned long long ctx = current_context_id();
    const SetupKey key{kern, ctx, threads, smem}, fkey{kern, ctx, 0, 0};
    std::lock_guard<std::mutex> lock(g_setup_mu);
    // The shared-memory limit is one value per kernel: raise it when a launch
    // needs more than has been set in this context, never lower it.
    auto lim = g_smem_limit.find(fkey);
    if (!ctx || lim == g_smem_limit.end() || lim->second < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (ctx) g_smem_limit[fkey] = smem;
    }
    if (!per_sm) return cudaSuccess;
    auto it = g_occupancy.find(key);
    if (ctx && it != g_occupancy.end()) {
        *per_sm = it->second;
        return cudaSuccess;
    }
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (ctx) g_occupancy[key] = n;
    *per_sm = n;
    return cudaSuccess;
}

int plan_sms(bool launch) { return launch ? std::min(sm_count(), kPlanMaxSms) : kPlanMaxSms; }

int plan_smem_per_sm(bool launch) {
    if (!launch) return kPlanMaxSmemPerSm;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kPlanMaxSmemPerSm;
    int v = g_smem_per_sm[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess || v <= 0)
            v = kPlanMaxSmemPerSm;
        g_smem_per_sm[dev].store(v, std::memory_order_relaxed);
    }
    return std::min(v, kPlanMaxSmemPerSm);
}

namespace {

long long floor_div(long long a, long long b) {  // b > 0
    long long q = a / b;
    if ((a % b != 0) && (a < 0)) --q;
    return q;
}

long long out_extent(long long X, long long F, long long S, long long D, long long P) {
    return floor_div(X + 2 * P - D * (F - 1) - 1, S) + 1;
}

int gcd(int a, int b) {
    while (b) {
        int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Validates sizes and fills the shape (OH, OW >= 1).  Elements per tensor are
// bounded so that every offset fits comfortably in 64-bit arithmetic.
dwconv_status make_shape(int N, int H, int W, int C, int FH, int FW, int SH, int SW, int DH, int DW, int PH,
                         int PW, Shape &s) {
    if (N <= 0 || H <= 0 || W <= 0 || C <= 0 || FH <= 0 || FW <= 0 || SH <= 0 || SW <= 0 || DH <= 0 ||
        DW <= 0 || PH < 0 || PW < 0)
        return DWCONV_ERR_INVALID_ARG;
    const long long OH = out_extent(H, FH, SH, DH, PH), OW = out_extent(W, FW, SW, DW, PW);
    if (OH < 1 || OW < 1 || OH > INT_MAX || OW > INT_MAX) return DWCONV_ERR_INVALID_ARG;
    const long long limit = 1LL << 40;
    if ((long long)N * H * W > limit / C || (long long)N * OH * OW > limit / C ||
        (long long)FH * FW > limit / C)
        return DWCONV_ERR_INVALID_ARG;
    s = Shape{N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW, (int)OH, (int)OW};
    return DWCONV_OK;
}

bool valid_dtype(dwconv_dtype dt) { return dt >= DWCONV_INT8 && dt <= DWCONV_FP8_E4M3; }

size_t elem_size(dwconv_dtype dt) {
    switch (dt) {
        case DWCONV_INT8: return 1;
        case DWCONV_FP8_E4M3: return 1;
        case DWCONV_FP32: return 4;
        default: return 2;
    }
}

// Element size of the forward output: int32 for int8 data, bf16 for FP8.
size_t out_elem_size(dwconv_dtype dt) {
    return dt == DWCONV_INT8 ? 4 : dt == DWCONV_FP8_E4M3 ? 2 : elem_size(dt);
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

dwconv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DWCONV_OK : DWCONV_ERR_CUDA; }

// Tiled kernels stage 16-byte copies of 32-channel slabs and store channel
// pairs: they need every pixel row to be a whole number of 16-byte copies.
bool tiled_layout_ok(const Shape &s, dwconv_dtype dt, const void *in, const void *out, const void *w) {
    if (dt == DWCONV_INT8) return false;
    const size_t es = elem_size(dt);
    if ((s.C * es) % 16 != 0) return false;
    return aligned(in, 16) && aligned(out, 2 * out_elem_size(dt)) && aligned(w, 2 * es);
}

// Taps read the input rows oh*SH - PH + fh*DH.  With g = gcd(SH, DH) they all
// lie in one residue class r0 = (-PH) mod g, so along H the pass is a stride
// SH/g, dilation DH/g convolution over that sub-grid (columns alike).  When
// both axes have unit stride and dilation on their sub-grids, fills the input
// side of p (the sub-grid and its padding) and returns true.  This covers the
// stride-2 dilation-2 layer, which reads only even rows and columns.
bool unit_subgrid(const Shape &s, TiledConv &p) {
    const int gh = gcd(s.SH, s.DH), gw = gcd(s.SW, s.DW);
    const int rh = (gh - s.PH % gh) % gh, rw = (gw - s.PW % gw) % gw;
    if (s.SH / gh != 1 || s.DH / gh != 1 || s.SW / gw != 1 || s.DW / gw != 1 || s.H <= rh || s.W <= rw)
        return false;
    p.Hf = s.H; p.Wf = s.W;
    p.in_step_h = gh; p.in_step_w = gw; p.in_off_h = rh; p.in_off_w = rw;
    p.Hs = (s.H - rh + gh - 1) / gh; p.Ws = (s.W - rw + gw - 1) / gw;
    p.pad_h = (s.PH + rh) / gh; p.pad_w = (s.PW + rw) / gw;
    return true;
}

// Strip filters taller than wide (FW < 8 <= FH, e.g. 51 x 5 or 31 x 1): the
// large-filter kernels walk filter rows and tile filter columns, so they take
// the problem transposed -- rows and columns exchange roles in the kernel's
// view (TiledConv::transpose) while the tensors stay where they are.
cudaError_t launch_tall_strip(const TiledConv &p, dwconv_dtype dt, cudaStream_t st) {
    if (!(p.FW < 8 && p.FH >= 8) || p.zero_phases || p.out_step_h != 1 || p.out_step_w != 1)
        return cudaErrorNotSupported;
    TiledConv q = p;
    q.transpose = 1;
    std::swap(q.Hs, q.Ws);
    std::swap(q.pad_h, q.pad_w);
    std::swap(q.FH, q.FW);
    std::swap(q.OHs, q.OWs);
    cudaError_t e = launch_tiled_mma_large(q, dt, st);
    if (e == cudaErrorNotSupported) e = launch_tiled_large(q, dt, st);
    return e;
}

// wgrad split of the direct path: slices of the N*OH*OW axis.  With
// launch = false a pure function of the shape, so that the workspace size can
// be computed without a device; a launch plans for the current device's SMs
// (never more slices than the workspace holds).
int wgrad_slices(const Shape &s, bool launch) {
    const long long positions = (long long)s.N * s.OH * s.OW;
    const long long per_slice_blocks = (long long)((s.C + 31) / 32) * s.FH * s.FW;
    const long long blocks = 8LL * plan_sms(launch);                  // ~8 blocks per SM
    long long z = (blocks + per_slice_blocks - 1) / per_slice_blocks;
    long long zmax = positions / 256;                                 // >= 256 positions a slice
    if (zmax < 1) zmax = 1;
    if (z > zmax) z = zmax;
    if (z > 4096) z = 4096;
    if (z < 1) z = 1;
    return (int)z;
}

// The weight gradient reads x on the same sub-grid as the forward pass; when
// that sub-grid has unit stride and dilation (and the channel rows are whole
// 16-byte copies) the tiled kernel can take it.  Shape-only: pointers may be
// null when only the plan is wanted.
bool wgrad_tiled_params(const Shape &s, dwconv_dtype dt, const void *x, const void *dy, float *dw,
                        TiledConv &p) {
    if (dt == DWCONV_INT8 || (s.C * elem_size(dt)) % 16 != 0) return false;
    p = TiledConv{};
    if (!unit_subgrid(s, p)) return false;
    p.in = x; p.w = nullptr; p.bias = nullptr; p.out = dw; p.dy = dy;
    p.N = s.N; p.C = s.C; p.FH = s.FH; p.FW = s.FW; p.flip = 0;
    p.OHf = s.OH; p.OWf = s.OW; p.OHs = s.OH; p.OWs = s.OW;
    p.out_step_h = p.out_step_w = 1; p.out_off_h = p.out_off_w = 0; p.zero_phases = 0;
    return true;
}

// The large-filter weight gradient walks filter columns in register windows:
// a filter taller than wide is taken transposed (TiledConv::transpose).
TiledConv wgrad_large_view(const TiledConv &p) {
    TiledConv q = p;
    if (p.FW < 8 && p.FH > p.FW) {
        q.transpose = 1;
        std::swap(q.Hs, q.Ws);
        std::swap(q.pad_h, q.pad_w);
        std::swap(q.FH, q.FW);
        std::swap(q.OHs, q.OWs);
    }
    return q;
}

// Slices (workspace) of the tiled weight-gradient path for this shape, 0 if none.
int wgrad_tiled_plan(const TiledConv &p, dwconv_dtype dt) {
    const int z = tiled_wgrad_slices(p, dt);
    if (z > 0) return z;
    const TiledConv q = wgrad_large_view(p);
    return std::max(tiled_mma_wgrad_slices(q, dt), tiled_wgrad_large_slices(q, dt));
}

}  // namespace
}  // namespace dwc

using namespace dwc;

extern "C" {

dwconv_status dwconv_output_size_2d(int H, int W, int FH, int FW, int stride_h, int stride_w, int dilation_h,
                                    int dilation_w, int pad_h, int pad_w, int *OH, int *OW) {
    Shape s;
    dwconv_status st = make_shape(1, H, W, 1, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, s);
    if (st != DWCONV_OK) return st;
    if (OH) *OH = s.OH;
    if (OW) *OW = s.OW;
    return DWCONV_OK;
}

dwconv_status dwconv_output_size(int H, int W, int FH, int FW, int stride, int dilation, int pad, int *OH,
                                 int *OW) {
    return dwconv_output_size_2d(H, W, FH, FW, stride, stride, dilation, dilation, pad, pad, OH, OW);
}

const char *dwconv_status_string(dwconv_status status) {
    switch (status) {
        case DWCONV_OK: return "DWCONV_OK";
        case DWCONV_ERR_INVALID_ARG: return "DWCONV_ERR_INVALID_ARG: invalid size, pointer or workspace";
        case DWCONV_ERR_UNSUPPORTED: return "DWCONV_ERR_UNSUPPORTED: dtype not provided for this pass";
        case DWCONV_ERR_MISALIGNED: return "DWCONV_ERR_MISALIGNED: pointer not aligned to its element size";
        case DWCONV_ERR_CUDA: return "DWCONV_ERR_CUDA: a CUDA call or kernel launch failed";
        case DWCONV_ERR_TIMEOUT: return "DWCONV_ERR_TIMEOUT: a bounded device wait gave up";
        default: return "unknown dwconv_status";
    }
}

unsigned long long dwconv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *dwconv_last_kernel(void) { return dwc::t_last_kernel; }

dwconv_status dwconv_check_device_errors(dwconv_stream stream) {
    unsigned v = 0;
    if (take_device_error(reinterpret_cast<cudaStream_t>(stream), &v) != cudaSuccess) return DWCONV_ERR_CUDA;
    return v ? DWCONV_ERR_TIMEOUT : DWCONV_OK;
}

}  // extern "C"

namespace dwc {
namespace {

dwconv_status fwd_impl(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w, int dilation_h,
                       int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype, const void *x, const void *w,
                       const void *bias, void *y, const Fuse &fz, dwconv_stream stream) {
    if (!valid_dtype(dtype)) return DWCONV_ERR_INVALID_ARG;
    Shape s;
    dwconv_status st =
        make_shape(N, H, W, C, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, s);
    if (st != DWCONV_OK) return st;
    if (!x || !w || !y) return DWCONV_ERR_INVALID_ARG;
    auto act_ok = [](int a) { return a >= DWCONV_ACT_NONE && a <= DWCONV_ACT_GELU; };
    if (!act_ok(fz.in_act) || !act_ok(fz.out_act)) return DWCONV_ERR_INVALID_ARG;
    if (dtype == DWCONV_INT8 && (fz.pre() || fz.post())) return DWCONV_ERR_UNSUPPORTED;
    if (dtype == DWCONV_FP8_E4M3 && fz.pre()) return DWCONV_ERR_UNSUPPORTED;
    const size_t es = elem_size(dtype);
    const size_t bs = 4;  // int32 (int8 data) or float bias
    const size_t ys = out_elem_size(dtype);
    if (!aligned(x, es) || !aligned(w, es) || !aligned(y, ys) || (bias && !aligned(bias, bs)))
        return DWCONV_ERR_MISALIGNED;
    for (const float *v : {fz.in_scale, fz.in_shift, fz.out_scale, fz.out_shift})
        if (v && !aligned(v, 4)) return DWCONV_ERR_MISALIGNED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

    // Unit stride and dilation on the taps' sub-grid (unit_subgrid) go to the
    // tiled kernels.  A kernel that does not provide a requested fusion
    // declines it (cudaErrorNotSupported) and the next one is tried.
    TiledConv p{};
    if (tiled_layout_ok(s, dtype, x, y, w) && unit_subgrid(s, p)) {
        p.in = x; p.w = w; p.bias = static_cast<const float *>(bias); p.out = y;
        p.N = N; p.C = C; p.FH = FH; p.FW = FW; p.flip = 0;
        p.OHf = s.OH; p.OWf = s.OW; p.OHs = s.OH; p.OWs = s.OW;
        p.out_step_h = p.out_step_w = 1; p.out_off_h = p.out_off_w = 0; p.zero_phases = 0;
        p.fz = fz;
        cudaError_t e = launch_tall_strip(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_mma(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_mma_large(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_smallmap(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_small(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_large(p, dtype, cs);
        if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    // Stride 2, dilation 1 (not a unit-stride sub-grid): the strided kernel
    // (plain or fused).
    if (tiled_layout_ok(s, dtype, x, y, w)) {
        cudaError_t e = launch_strided_fwd(s, dtype, x, w, static_cast<const float *>(bias), y, fz, cs);
        if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    return cuda_status(launch_fwd_direct(s, dtype, x, w, bias, y, fz, cs));
}

}  // namespace
}  // namespace dwc

extern "C" {

dwconv_status dwconv_fwd_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                            int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype, const void *x,
                            const void *w, const void *bias, void *y, dwconv_stream stream) {
    return fwd_impl(N, H, W, C, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, dtype, x, w,
                    bias, y, Fuse{}, stream);
}

dwconv_status dwconv_fwd_fused_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                                  int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                                  const void *x, const float *in_scale, const float *in_shift,
                                  dwconv_activation in_act, const void *w, const void *bias,
                                  const float *out_scale, const float *out_shift, dwconv_activation out_act,
                                  void *y, dwconv_stream stream) {
    const Fuse fz{in_scale, in_shift, (int)in_act, out_scale, out_shift, (int)out_act};
    return fwd_impl(N, H, W, C, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, dtype, x, w,
                    bias, y, fz, stream);
}

dwconv_status dwconv_fwd_fused(int N, int H, int W, int C, int FH, int FW, int stride, int dilation, int pad,
                               dwconv_dtype dtype, const void *x, const float *in_scale, const float *in_shift,
                               dwconv_activation in_act, const void *w, const void *bias, const float *out_scale,
                               const float *out_shift, dwconv_activation out_act, void *y, dwconv_stream stream) {
    return dwconv_fwd_fused_2d(N, H, W, C, FH, FW, stride, stride, dilation, dilation, pad, pad, dtype, x,
                               in_scale, in_shift, in_act, w, bias, out_scale, out_shift, out_act, y, stream);
}

dwconv_status dwconv_fwd(int N, int H, int W, int C, int FH, int FW, int stride, int dilation, int pad,
                         dwconv_dtype dtype, const void *x, const void *w, const void *bias, void *y,
                         dwconv_stream stream) {
    return dwconv_fwd_2d(N, H, W, C, FH, FW, stride, stride, dilation, dilation, pad, pad, dtype, x, w, bias, y,
                         stream);
}

dwconv_status dwconv_bwd_data_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                                 int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                                 const void *dy, const void *w, void *dx, dwconv_stream stream) {
    if (!valid_dtype(dtype)) return DWCONV_ERR_INVALID_ARG;
    Shape s;
    dwconv_status st =
        make_shape(N, H, W, C, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, s);
    if (st != DWCONV_OK) return st;
    if (dtype == DWCONV_INT8 || dtype == DWCONV_FP8_E4M3) return DWCONV_ERR_UNSUPPORTED;
    if (!dy || !w || !dx) return DWCONV_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (!aligned(dy, es) || !aligned(w, es) || !aligned(dx, es)) return DWCONV_ERR_MISALIGNED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

    // When S divides D (per axis), every tap of input row ih satisfies
    // ih = S*i + ph with ph = (-P) mod S, and dx on that phase is a unit-stride
    // convolution of dy with the filter rotated by 180 degrees (Flash-DWC §5.1,
    // generalised from S = 1), dilation D/S and padding (F-1)*D/S - (ph+P)/S;
    // every other phase receives no tap and is written as zero.
    const int SH = stride_h, SW = stride_w;
    if (dilation_h % SH == 0 && dilation_h / SH == 1 && dilation_w % SW == 0 && dilation_w / SW == 1 &&
        tiled_layout_ok(s, dtype, dy, dx, w)) {
        const int phh = (SH - pad_h % SH) % SH, phw = (SW - pad_w % SW) % SW;
        const int qh = (phh + pad_h) / SH, qw = (phw + pad_w) / SW;
        TiledConv p{};
        p.in = dy; p.w = w; p.bias = nullptr; p.out = dx;
        p.N = N; p.C = C; p.FH = FH; p.FW = FW; p.flip = 1;
        p.Hf = s.OH; p.Wf = s.OW; p.Hs = s.OH; p.Ws = s.OW;
        p.in_step_h = p.in_step_w = 1; p.in_off_h = p.in_off_w = 0;
        p.pad_h = (FH - 1) * (dilation_h / SH) - qh;
        p.pad_w = (FW - 1) * (dilation_w / SW) - qw;
        p.OHf = H; p.OWf = W;
        p.OHs = (H + SH - 1) / SH; p.OWs = (W + SW - 1) / SW;
        p.out_step_h = SH; p.out_step_w = SW; p.out_off_h = phh; p.out_off_w = phw;
        p.zero_phases = (SH > 1 || SW > 1) ? 1 : 0;
        if (p.zero_phases) {
            // Tensor-core kernel on the one live phase (its exact extent, so the
            // TMA store stays inside dx); the other phases are zeroed first.
            TiledConv pm = p;
            pm.zero_phases = 0;
            pm.OHs = (H - phh + SH - 1) / SH;
            pm.OWs = (W - phw + SW - 1) / SW;
            if (pm.OHs > 0 && pm.OWs > 0 && tiled_mma_supports(pm, dtype)) {
                cudaError_t e = cudaMemsetAsync(dx, 0, (size_t)N * H * W * C * es, cs);
                if (e != cudaSuccess) return DWCONV_ERR_CUDA;
                e = launch_tiled_mma(pm, dtype, cs);
                if (e != cudaErrorNotSupported) return cuda_status(e);
            }
        }
        cudaError_t e = launch_tall_strip(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_mma(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_mma_large(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_smallmap(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_small(p, dtype, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_large(p, dtype, cs);
        if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    // Stride 2, dilation 1: all four output phases of dx in one strided kernel.
    if (tiled_layout_ok(s, dtype, dy, dx, w)) {
        cudaError_t e = launch_strided_dgrad(s, dtype, dy, w, dx, cs);
        if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    return cuda_status(launch_dgrad_direct(s, dtype, dy, w, dx, cs));
}

dwconv_status dwconv_bwd_data(int N, int H, int W, int C, int FH, int FW, int stride, int dilation, int pad,
                              dwconv_dtype dtype, const void *dy, const void *w, void *dx, dwconv_stream stream) {
    return dwconv_bwd_data_2d(N, H, W, C, FH, FW, stride, stride, dilation, dilation, pad, pad, dtype, dy, w, dx,
                              stream);
}

size_t dwconv_bwd_filter_workspace_size_2d(int N, int H, int W, int C, int FH, int FW, int stride_h,
                                           int stride_w, int dilation_h, int dilation_w, int pad_h, int pad_w,
                                           dwconv_dtype dtype) {
    Shape s;
    if (!valid_dtype(dtype) || dtype == DWCONV_INT8 || dtype == DWCONV_FP8_E4M3) return 0;
    if (make_shape(N, H, W, C, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, s) != DWCONV_OK)
        return 0;
    const size_t per_slice = (size_t)FH * FW * C * sizeof(float);
    size_t need = (size_t)wgrad_slices(s, false) * per_slice;
    TiledConv p;
    if (wgrad_tiled_params(s, dtype, nullptr, nullptr, nullptr, p)) {
        const size_t tiled = (size_t)wgrad_tiled_plan(p, dtype) * per_slice;
        if (tiled > need) need = tiled;
        need = std::max(need, (size_t)smallmap_wgrad_slices(p, dtype) * per_slice);
    }
    need = std::max(need, (size_t)strided_wgrad_slices(s, dtype) * per_slice);
    return need;
}

size_t dwconv_bwd_filter_workspace_size(int N, int H, int W, int C, int FH, int FW, int stride, int dilation,
                                        int pad, dwconv_dtype dtype) {
    return dwconv_bwd_filter_workspace_size_2d(N, H, W, C, FH, FW, stride, stride, dilation, dilation, pad, pad,
                                               dtype);
}

}  // extern "C"

namespace dwc {
namespace {

dwconv_status bwd_filter_impl(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                              int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                              const void *x, const void *dy, float *dw, void *workspace, size_t workspace_bytes,
                              int half_accumulate, dwconv_stream stream) {
    if (!valid_dtype(dtype)) return DWCONV_ERR_INVALID_ARG;
    Shape s;
    dwconv_status st =
        make_shape(N, H, W, C, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, s);
    if (st != DWCONV_OK) return st;
    if (dtype == DWCONV_INT8 || dtype == DWCONV_FP8_E4M3 || (half_accumulate && dtype != DWCONV_FP16))
        return DWCONV_ERR_UNSUPPORTED;
    if (!x || !dy || !dw) return DWCONV_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (!aligned(x, es) || !aligned(dy, es) || !aligned(dw, 4)) return DWCONV_ERR_MISALIGNED;
    const size_t need = dwconv_bwd_filter_workspace_size_2d(N, H, W, C, FH, FW, stride_h, stride_w,
                                                            dilation_h, dilation_w, pad_h, pad_w, dtype);
    if (workspace_bytes < need || (need > 0 && !workspace)) return DWCONV_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return DWCONV_ERR_MISALIGNED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    float *part = static_cast<float *>(workspace);

    TiledConv p;
    if (wgrad_tiled_params(s, dtype, x, dy, dw, p) && aligned(x, 16) && aligned(dy, 16)) {
        p.half_accumulate = half_accumulate;
        cudaError_t e = launch_smallmap_wgrad(p, dtype, part, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_wgrad(p, dtype, part, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_mma_wgrad(wgrad_large_view(p), dtype, part, cs);
        if (e == cudaErrorNotSupported) e = launch_tiled_wgrad_large(wgrad_large_view(p), dtype, part, cs);
        if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    if ((s.C * es) % 16 == 0 && aligned(x, 16) && aligned(dy, 16)) {
        cudaError_t e = launch_strided_wgrad(s, dtype, x, dy, part, dw, cs);
        if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    // Shapes without a tiled instance take the exact fp32 path, also for the
    // hybrid-accumulation entry point (its bound holds a fortiori).
    const int Z = wgrad_slices(s, true);
    cudaError_t e = launch_wgrad_direct(s, dtype, x, dy, part, Z, cs);
    if (e != cudaSuccess) return DWCONV_ERR_CUDA;
    return cuda_status(launch_wgrad_reduce(part, Z, (long long)FH * FW * C, dw, cs));
}

}  // namespace
}  // namespace dwc

extern "C" {

dwconv_status dwconv_bwd_filter_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                                   int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                                   const void *x, const void *dy, float *dw, void *workspace,
                                   size_t workspace_bytes, dwconv_stream stream) {
    return bwd_filter_impl(N, H, W, C, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, dtype, x,
                           dy, dw, workspace, workspace_bytes, 0, stream);
}

dwconv_status dwconv_bwd_filter_ha_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                                      int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                                      const void *x, const void *dy, float *dw, void *workspace,
                                      size_t workspace_bytes, dwconv_stream stream) {
    return bwd_filter_impl(N, H, W, C, FH, FW, stride_h, stride_w, dilation_h, dilation_w, pad_h, pad_w, dtype, x,
                           dy, dw, workspace, workspace_bytes, 1, stream);
}

dwconv_status dwconv_bwd_filter_ha(int N, int H, int W, int C, int FH, int FW, int stride, int dilation, int pad,
                                   dwconv_dtype dtype, const void *x, const void *dy, float *dw, void *workspace,
                                   size_t workspace_bytes, dwconv_stream stream) {
    return dwconv_bwd_filter_ha_2d(N, H, W, C, FH, FW, stride, stride, dilation, dilation, pad, pad, dtype, x, dy,
                                   dw, workspace, workspace_bytes, stream);
}

dwconv_status dwconv_bwd_filter(int N, int H, int W, int C, int FH, int FW, int stride, int dilation, int pad,
                                dwconv_dtype dtype, const void *x, const void *dy, float *dw, void *workspace,
                                size_t workspace_bytes, dwconv_stream stream) {
    return dwconv_bwd_filter_2d(N, H, W, C, FH, FW, stride, stride, dilation, dilation, pad, pad, dtype, x, dy, dw,
                                workspace, workspace_bytes, stream);
}

size_t dwconv_bwd_bias_workspace_size(int N, int OH, int OW, int C) {
    if (N < 1 || OH < 1 || OW < 1 || C < 1) return 0;
    const long long P = (long long)N * OH * OW;
    if (P > (1LL << 40) || (long long)C * P > (1LL << 50)) return 0;
    return (size_t)bias_slices(P, C, false) * (size_t)C * sizeof(float);
}

dwconv_status dwconv_bwd_bias(int N, int OH, int OW, int C, dwconv_dtype dtype, const void *dy, float *db,
                              void *workspace, size_t workspace_bytes, dwconv_stream stream) {
    if (!valid_dtype(dtype)) return DWCONV_ERR_INVALID_ARG;
    const size_t need = dwconv_bwd_bias_workspace_size(N, OH, OW, C);
    if (need == 0) return DWCONV_ERR_INVALID_ARG;
    if (dtype == DWCONV_INT8 || dtype == DWCONV_FP8_E4M3) return DWCONV_ERR_UNSUPPORTED;
    if (!dy || !db || !workspace || workspace_bytes < need) return DWCONV_ERR_INVALID_ARG;
    if (!aligned(dy, elem_size(dtype)) || !aligned(db, 4) || !aligned(workspace, 16)) return DWCONV_ERR_MISALIGNED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const long long P = (long long)N * OH * OW;
    const int Z = bias_slices(P, C, true);
    float *part = static_cast<float *>(workspace);
    cudaError_t e = launch_bias_slices(P, C, dtype, dy, part, Z, cs);
    if (e != cudaSuccess) return cuda_status(e);
    return cuda_status(launch_wgrad_reduce(part, Z, C, db, cs));
}

}  // extern "C"
