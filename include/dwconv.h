/*
 * dwconv.h - C ABI of libdwconv, depthwise 2-D convolution on one GB300 (sm_103a).
 *
 * The operation ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on
 * GPUs", §2.1 "Standard and depthwise convolution", Fig. 1; layouts from §2.3
 * "Unified channels-last layout"): every channel c has its own FH x FW filter,
 *
 *   y[n,oh,ow,c] = bias[c] + sum_{fh<FH, fw<FW} w[fh,fw,c] * x[n, oh*S-P+fh*D, ow*S-P+fw*D, c]
 *
 * where x positions outside [0,H) x [0,W) read as zero (padding is generated,
 * never fetched: "Tiles, halos and partial sums", "Partition tensors to fit
 * storage").  S = stride, D = dilation, P = pad, the same along both axes.
 * Output size (floor convention):
 *
 *   OH = floor((H + 2P - D(FH-1) - 1) / S) + 1,   OW likewise.
 *
 * Layouts (all dense, row-major, channels innermost):
 *   x, dx   [N][H][W][C]      y, dy  [N][OH][OW][C]
 *   w       [FH][FW][C]       dw     [FH][FW][C] (fp32)     bias [C]
 *
 * Element types per dtype:
 *   DWCONV_INT8  x, w int8;  bias int32 (nullable); y int32.  Forward only.
 *                Accumulation in int32; overflow wraps (two's complement).
 *   DWCONV_FP32  x, w, bias, y, dy, dx, dw: float.
 *   DWCONV_FP16  x, w, y, dy, dx: IEEE half; bias, dw: float.
 *   DWCONV_BF16  x, w, y, dy, dx: bfloat16;  bias, dw: float.
 *   DWCONV_FP8_E4M3  x, w: OCP FP8 E4M3 (1 sign, 4 exponent bits with bias 7,
 *                3 mantissa bits, no infinities, NaN = S.1111.111, largest
 *                448); bias float; y bfloat16.  Forward pass only
 *                (dwconv_fwd*, the fused form with an epilogue but no
 *                prologue); every other entry point returns
 *                DWCONV_ERR_UNSUPPORTED.  Operands widen exactly to fp32; a
 *                per-tensor or per-channel dequantisation scale folds into
 *                the fused epilogue's out_scale.  (The pages name low-bit
 *                types such as FP8 as an extension: stored and multiplied in
 *                low precision, accumulated in fp32.)
 *   Floating-point accumulation is fp32 in every case (Flash-DWC §4.1 shows
 *   16-bit accumulation loses too much accuracy); 16-bit outputs are rounded
 *   to nearest even once, at the end.
 *
 * Ownership and ordering: the caller owns every buffer (device memory, e.g.
 * from PyTorch); the library allocates no device memory, keeps no per-call
 * state and caches only device properties.  Every call validates its
 * arguments on the host, then enqueues kernels on `stream` and returns before
 * they finish (stream-ordered, like cudaMemcpyAsync).  Input buffers must not
 * overlap output buffers.
 *
 * Errors: status codes only.  Validation happens before any launch; on a
 * non-OK status nothing was enqueued.  A launch failure returns
 * DWCONV_ERR_CUDA; faults that happen later surface on the stream as usual.
 */
#ifndef DWCONV_H
#define DWCONV_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DWCONV_OK = 0,
    DWCONV_ERR_INVALID_ARG = 1,  /* bad size, null pointer, empty output, small workspace */
    DWCONV_ERR_UNSUPPORTED = 2,  /* dtype/pass pair not provided (int8 backward) */
    DWCONV_ERR_MISALIGNED = 3,   /* a pointer not aligned to its element size */
    DWCONV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    DWCONV_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up (see dwconv_check_device_errors) */
} dwconv_status;

typedef enum {
    DWCONV_INT8 = 0,
    DWCONV_FP32 = 1,
    DWCONV_FP16 = 2,
    DWCONV_BF16 = 3,
    DWCONV_FP8_E4M3 = 4
} dwconv_dtype;

/* Activation functions of the fused forward pass (dwconv_fwd_fused). */
typedef enum {
    DWCONV_ACT_NONE = 0,   /* identity */
    DWCONV_ACT_RELU = 1,   /* max(v, 0) */
    DWCONV_ACT_RELU6 = 2,  /* min(max(v, 0), 6) */
    DWCONV_ACT_SILU = 3,   /* v * sigmoid(v) = v / (1 + exp(-v)) */
    DWCONV_ACT_GELU = 4    /* v * Phi(v) = v/2 * (1 + erf(v / sqrt 2)), the exact (erf) form */
} dwconv_activation;

/* A CUDA stream (the same handle as cudaStream_t).  NULL = the legacy default stream. */
typedef struct CUstream_st *dwconv_stream;

/*
 * Output extent of the forward pass for an H x W input (floor convention above).
 * Writes *OH and *OW (either may be NULL).  Returns DWCONV_ERR_INVALID_ARG if a size
 * or S, D is non-positive, P is negative, or the output would be empty.
 */
dwconv_status dwconv_output_size(int H, int W, int FH, int FW, int stride, int dilation, int pad,
                                 int *OH, int *OW);

/*
 * Forward pass (Flash-DWC §5.1 "FC"): y = DWC(x, w) + bias.
 * x [N][H][W][C], w [FH][FW][C], bias [C] or NULL (no bias), y [N][OH][OW][C].
 * The bias enters each output exactly once ("Tiles, halos and partial sums":
 * partial sums keep full precision across tiles and the bias is added once).
 */
dwconv_status dwconv_fwd(int N, int H, int W, int C, int FH, int FW, int stride, int dilation,
                         int pad, dwconv_dtype dtype, const void *x, const void *w,
                         const void *bias, void *y, dwconv_stream stream);

/*
 * Input gradient (Flash-DWC §5.1 "BDC"): dx = the adjoint of the bias-free
 * forward map applied to dy, i.e.
 *   dx[n,ih,iw,c] = sum over (oh,ow,fh,fw) with oh*S-P+fh*D = ih and
 *                   ow*S-P+fw*D = iw of w[fh,fw,c] * dy[n,oh,ow,c].
 * For S = 1 this is the forward pass over dy with the filter rotated by 180
 * degrees and padding D(FH-1)-P, as §5.1 states; for S > 1 positions that no
 * tap reaches receive 0.  dy [N][OH][OW][C] (OH, OW of an H x W input),
 * w [FH][FW][C], dx [N][H][W][C] (every element written).  fp32, fp16 and bf16;
 * DWCONV_INT8 and DWCONV_FP8_E4M3 return DWCONV_ERR_UNSUPPORTED.
 */
dwconv_status dwconv_bwd_data(int N, int H, int W, int C, int FH, int FW, int stride,
                              int dilation, int pad, dwconv_dtype dtype, const void *dy,
                              const void *w, void *dx, dwconv_stream stream);

/*
 * Bytes of device scratch that dwconv_bwd_filter needs for this shape (the
 * per-slice partial sums of the split reduction).  A pure function of the
 * arguments; 0 if they are invalid.
 */
size_t dwconv_bwd_filter_workspace_size(int N, int H, int W, int C, int FH, int FW, int stride,
                                        int dilation, int pad, dwconv_dtype dtype);

/*
 * Weight gradient (Flash-DWC §5.1 "BFC"):
 *   dw[fh,fw,c] = sum over (n,oh,ow) with the tap inside the input of
 *                 dy[n,oh,ow,c] * x[n, oh*S-P+fh*D, ow*S-P+fw*D, c].
 * The N*OH*OW accumulation axis is split into slices reduced in parallel and
 * then summed in a fixed order (§5.1 "accumulation-axis parallelisation"), so
 * repeated calls give bit-identical dw.  x [N][H][W][C], dy [N][OH][OW][C],
 * dw [FH][FW][C] float (fully overwritten).  `workspace` is caller-owned
 * device memory of at least dwconv_bwd_filter_workspace_size() bytes, 16-byte
 * aligned (else DWCONV_ERR_MISALIGNED); it may be NULL only if that size is 0.  fp32, fp16 and bf16 only
 * (DWCONV_INT8 and DWCONV_FP8_E4M3: DWCONV_ERR_UNSUPPORTED, workspace size 0).
 */
dwconv_status dwconv_bwd_filter(int N, int H, int W, int C, int FH, int FW, int stride,
                                int dilation, int pad, dwconv_dtype dtype, const void *x,
                                const void *dy, float *dw, void *workspace,
                                size_t workspace_bytes, dwconv_stream stream);

/*
 * Bytes of device scratch that dwconv_bwd_bias needs (per-slice partial sums).
 * A pure function of the arguments; 0 if they are invalid.
 */
size_t dwconv_bwd_bias_workspace_size(int N, int OH, int OW, int C);

/*
 * Bias gradient: db[c] = sum over (n,oh,ow) of dy[n,oh,ow,c], the adjoint of
 * adding bias[c] once to every output (Flash-DWC §5.1's training passes stop
 * at the input and weight gradients; a layer with a bias needs this one too).
 * dy [N][OH][OW][C]
 * in the pass's dtype, db [C] float (fully overwritten).  The N*OH*OW axis is
 * split into slices summed in parallel, then added in a fixed order, so
 * repeated calls give bit-identical db.  `workspace`: caller-owned device
 * memory of at least dwconv_bwd_bias_workspace_size() bytes, 16-byte aligned.
 * fp32, fp16 and bf16 only; DWCONV_INT8 and DWCONV_FP8_E4M3 return
 * DWCONV_ERR_UNSUPPORTED.
 */
dwconv_status dwconv_bwd_bias(int N, int OH, int OW, int C, dwconv_dtype dtype, const void *dy,
                              float *db, void *workspace, size_t workspace_bytes, dwconv_stream stream);

/* Bytes of device scratch built into the library for dwconv_bwd_filter_static. */
#define DWCONV_STATIC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * Weight gradient for callers that cannot allocate device memory.  The paper
 * has no counterpart: this is a deployment convenience of this library.
 *
 * Same operation, arguments and result as dwconv_bwd_filter, minus the
 * workspace.  It is for code that has no way to obtain scratch memory: for
 * example an operator running inside a framework whose caching allocator
 * already owns the device memory (so calling cudaMalloc would go around it),
 * or a deployment that fixes its memory plan at start-up and forbids
 * allocation afterwards.  The call allocates nothing; it uses a
 * DWCONV_STATIC_SCRATCH_BYTES array compiled into the library, which every
 * GPU that loads the library holds until the process exits.
 *
 * - Shapes whose dwconv_bwd_filter_workspace_size() exceeds
 *   DWCONV_STATIC_SCRATCH_BYTES are rejected with DWCONV_ERR_INVALID_ARG
 *   before anything is enqueued; use dwconv_bwd_filter for those.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture on the device.  The cached address
 *   belongs to the device's current context: after a device reset the first
 *   call in the new context looks it up again (so make that call, too, outside
 *   a stream capture).
 * - All calls on a device share the one array, and it keeps whatever the last
 *   call left in it.  Calls whose work overlaps on the GPU (different streams,
 *   no ordering between them) race on it and give wrong results: order them.
 *   Nothing in the array needs to start at zero; each call writes every
 *   partial sum before reading it.
 */
dwconv_status dwconv_bwd_filter_static(int N, int H, int W, int C, int FH, int FW, int stride,
                                       int dilation, int pad, dwconv_dtype dtype, const void *x,
                                       const void *dy, float *dw, dwconv_stream stream);

/*
 * Waits for `stream`, then reports whether any kernel of this library on the
 * current device gave up a bounded wait since the last check: the kernels
 * that stage tiles with TMA wait on shared-memory barriers for a bounded
 * number of polls (seconds), and on running out they record the fact and
 * return instead of hanging.  Returns DWCONV_ERR_TIMEOUT (and clears the
 * record) if that happened, DWCONV_ERR_CUDA if the stream reports an error,
 * DWCONV_OK otherwise.
 */
dwconv_status dwconv_check_device_errors(dwconv_stream stream);

/*
 * Self-test of that failure detection: enqueues on `stream` one thread that
 * waits, with a short bound (milliseconds), on a shared-memory barrier that
 * nothing completes -- the kind of wait the tiled kernels make for their
 * copies -- gives up and records the timeout as they would.  No fault, no
 * hang; caller memory is not touched.  The next dwconv_check_device_errors
 * returns DWCONV_ERR_TIMEOUT (and clears the record).  Returns DWCONV_OK once
 * enqueued, DWCONV_ERR_CUDA if the launch fails.
 */
dwconv_status dwconv_selftest_timeout(dwconv_stream stream);

/*
 * Per-axis forms.  Each _2d entry point is the operation of the entry point of
 * the same name with the stride, dilation and padding given separately for
 * the H and W axes: taps read x[n, oh*stride_h - pad_h + fh*dilation_h,
 * ow*stride_w - pad_w + fw*dilation_w, c], and
 * OH = floor((H + 2 pad_h - dilation_h (FH-1) - 1) / stride_h) + 1 (OW alike).
 * (The pages give one stride, dilation and padding; the per-axis form is the
 * same index formula per axis, needed e.g. for "same" padding of 1 x K strip
 * filters.)  Arguments, layouts, ownership, workspace and errors are those of
 * the symmetric entry points, which call these with equal values per axis.
 */
dwconv_status dwconv_output_size_2d(int H, int W, int FH, int FW, int stride_h, int stride_w, int dilation_h,
                                    int dilation_w, int pad_h, int pad_w, int *OH, int *OW);
dwconv_status dwconv_fwd_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                            int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype, const void *x,
                            const void *w, const void *bias, void *y, dwconv_stream stream);
dwconv_status dwconv_bwd_data_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                                 int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                                 const void *dy, const void *w, void *dx, dwconv_stream stream);
size_t dwconv_bwd_filter_workspace_size_2d(int N, int H, int W, int C, int FH, int FW, int stride_h,
                                           int stride_w, int dilation_h, int dilation_w, int pad_h, int pad_w,
                                           dwconv_dtype dtype);
dwconv_status dwconv_bwd_filter_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                                   int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                                   const void *x, const void *dy, float *dw, void *workspace,
                                   size_t workspace_bytes, dwconv_stream stream);

/*
 * Fused forward pass (Flash-DWC §5.2 "Kernel fusion": depthwise convolutions
 * usually sit next to a batch normalisation and an activation, BN+Act+DWC;
 * fusing them into the convolution's kernel saves the memory passes of the
 * separate layers).  BN in inference form is a per-channel affine map, so
 * with per-channel scale and shift vectors the pass computes
 *
 *   x'[n,ih,iw,c] = round_T(in_act(in_scale[c] * x[n,ih,iw,c] + in_shift[c]))
 *   z[n,oh,ow,c]  = bias[c] + sum w[fh,fw,c] * x'[n, oh*stride_h-pad_h+fh*dilation_h, ..., c]
 *   y[n,oh,ow,c]  = round_T(out_act(out_scale[c] * z[n,oh,ow,c] + out_shift[c]))
 *
 * with x' outside the input reading as zero (the padding belongs to x', the
 * tensor the unfused BN+Act layer would have written) and round_T the
 * rounding to the storage type (none for fp32): x' holds exactly what the
 * unfused layer would store.  The affine maps are one fp32 fused
 * multiply-add; the activations are evaluated in fp32 (SiLU with the fast
 * exponential and reciprocal, GELU through the erfc approximation of
 * Abramowitz & Stegun 7.1.26, |error| <= 1.5e-7: both within 1e-6 |v| + 1e-7
 * of the exact function).
 * in_scale, in_shift, out_scale, out_shift: float [C] device vectors, each
 * nullable (NULL scale = 1, NULL shift = 0); *_act a dwconv_activation.
 * With every one of them NULL / DWCONV_ACT_NONE the call is dwconv_fwd_2d.
 * Other arguments, layouts, ownership and errors as dwconv_fwd_2d; the
 * fused vectors must be 4-byte aligned (else DWCONV_ERR_MISALIGNED), an
 * activation outside the enum is DWCONV_ERR_INVALID_ARG, and DWCONV_INT8
 * with any fusion is DWCONV_ERR_UNSUPPORTED.
 */
dwconv_status dwconv_fwd_fused_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                                  int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                                  const void *x, const float *in_scale, const float *in_shift,
                                  dwconv_activation in_act, const void *w, const void *bias,
                                  const float *out_scale, const float *out_shift, dwconv_activation out_act,
                                  void *y, dwconv_stream stream);
/* dwconv_fwd_fused_2d with the same stride, dilation and padding on both axes. */
dwconv_status dwconv_fwd_fused(int N, int H, int W, int C, int FH, int FW, int stride, int dilation, int pad,
                               dwconv_dtype dtype, const void *x, const float *in_scale, const float *in_shift,
                               dwconv_activation in_act, const void *w, const void *bias, const float *out_scale,
                               const float *out_shift, dwconv_activation out_act, void *y, dwconv_stream stream);

/*
 * Weight gradient with hybrid accumulation (Flash-DWC §5.1 "mixed
 * accumulation", an opt-in): the long accumulation over N*OH*OW is split into
 * short sub-units, each summed in fp16, and the sub-unit sums are merged in
 * fp32.  Here a sub-unit is the products of one thread's output tile of one
 * work unit (14 positions per tap for 7x7 filters, 28 for 3x3 and 5x5),
 * accumulated with packed fp16 fused multiply-adds (two channels per
 * instruction).  Error bound per dw element: gamma_L * sum |dy * x| with
 * L <= 28 and fp16's unit roundoff u = 2^-11 (gamma_L = L u / (1 - L u),
 * 1.39e-2 for L = 28), plus the fp32 merge; every fp16 partial sum must stay
 * below 65504 in magnitude.
 * Arguments, workspace (dwconv_bwd_filter_workspace_size_2d), layouts and
 * errors as dwconv_bwd_filter_2d; DWCONV_FP16 only (other dtypes:
 * DWCONV_ERR_UNSUPPORTED).  Shapes the tiled weight-gradient kernel does not
 * cover run the exact fp32 path instead (dwconv_last_kernel says which ran:
 * "tiled_wgrad_ha" for the hybrid kernel).
 */
dwconv_status dwconv_bwd_filter_ha_2d(int N, int H, int W, int C, int FH, int FW, int stride_h, int stride_w,
                                      int dilation_h, int dilation_w, int pad_h, int pad_w, dwconv_dtype dtype,
                                      const void *x, const void *dy, float *dw, void *workspace,
                                      size_t workspace_bytes, dwconv_stream stream);
/* dwconv_bwd_filter_ha_2d with the same stride, dilation and padding on both axes. */
dwconv_status dwconv_bwd_filter_ha(int N, int H, int W, int C, int FH, int FW, int stride, int dilation, int pad,
                                   dwconv_dtype dtype, const void *x, const void *dy, float *dw, void *workspace,
                                   size_t workspace_bytes, dwconv_stream stream);

/* A static, human-readable name for a status code. */
const char *dwconv_status_string(dwconv_status status);

/*
 * Number of kernels this library has launched in this process (all threads,
 * all devices).  Lets a caller count launches over a region of interest.
 */
unsigned long long dwconv_launch_count(void);

/*
 * Kernel family of the latest pass this host thread launched, as a static
 * string: "tiled_mma" (tensor-core Toeplitz, 16-bit 3x3/5x5/7x7),
 * "tiled_mma_large" (tensor-core Toeplitz, large 16-bit filters),
 * "tiled_small" / "tiled_large" (register-tiled FMA kernels), "tiled_wgrad"
 * (tiled weight gradient), "tiled_wgrad_ha" (its hybrid-accumulation form),
 * "tiled_mma_wgrad" (tensor-core weight gradient, large 16-bit filters),
 * "tiled_wgrad_large" (tap-group weight gradient, other large filters), "direct_fwd" / "direct_dgrad" / "direct_wgrad"
 * (one output per thread), or "none" before the first launch.  The host-side
 * dispatch sets it when it launches; it says nothing about completion.  For
 * reporting which kernel ran (e.g. against which roofline to measure it).
 * No counterpart in the method's description: introspection only.
 */
const char *dwconv_last_kernel(void);

#ifdef __cplusplus
}
#endif

#endif /* DWCONV_H */
