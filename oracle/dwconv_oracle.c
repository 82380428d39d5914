/*
 * Depthwise 2-D convolution oracle: plain, slow, direct loops on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (Flash-DWC: Making Depthwise Convolution Compute-Efficient
 * on GPUs, §2.1 "Standard and depthwise convolution" and §2.3 "Unified
 * channels-last layout"): every channel c has its own FH x FW filter and
 *
 *   y[n,oh,ow,c] = bias[c] + sum_{fh<FH, fw<FW} w[fh,fw,c] * x[n, oh*S-P+fh*D, ow*S-P+fw*D, c]
 *
 * with x, y in NHWC, w in FH x FW x C, and x read as zero outside [0,H)x[0,W)
 * (zero padding: "Outline of Programming Massively Parallel Processors",
 * section "Convolution / 2D Convolution"; "Tiles, halos and partial sums",
 * "boundary padding may be generated").  The output size uses the floor
 * convention OH = floor((H + 2P - D(FH-1) - 1)/S) + 1.
 *
 * The two training passes of Flash-DWC §5.1 "Backward propagation":
 *   dgrad (BDC): dx = the exact adjoint of the bias-free forward map applied to
 *                dy, written here as the scatter dx[n,ih,iw,c] += w*dy over
 *                every (n,oh,ow,fh,fw) whose tap lands inside the input;
 *   wgrad (BFC): dw[fh,fw,c] = sum over (n,oh,ow) with the tap inside the
 *                input of dy[n,oh,ow,c] * x[n,ih,iw,c].
 *
 * Arithmetic: float64 for floating-point data (the caller passes the exact
 * 16/32-bit values widened to double), int64 for integer data.  Every
 * function also returns, per output element, the magnitude
 * mag = |bias| + sum |product| that the parity tolerance scales with.
 *
 * Each output element is accumulated in the order fh (outer), fw (inner) for
 * the forward pass, (n, oh, ow) for wgrad and (n, oh, ow, fh, fw) for the
 * dgrad scatter.  Work is split across threads by channel ranges only; every
 * output element is owned by exactly one thread, so results do not depend on
 * the thread count.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- shape ------------------------------------------------------------- */

typedef struct {
    long N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW, OH, OW;  /* stride, dilation, padding per axis */
} dwo_shape;

static long floor_div(long a, long b) { /* b > 0 */
    long q = a / b;
    if ((a % b != 0) && (a < 0)) q -= 1;
    return q;
}

/* Output extent along one axis: floor((X + 2P - D(F-1) - 1)/S) + 1. */
long dwo_out_extent(long X, long F, long S, long D, long P) {
    if (S <= 0 || D <= 0 || F <= 0) return 0;
    return floor_div(X + 2 * P - D * (F - 1) - 1, S) + 1;
}

static int make_shape(dwo_shape *s, long N, long H, long W, long C, long FH, long FW,
                      long SH, long SW, long DH, long DW, long PH, long PW) {
    if (N <= 0 || H <= 0 || W <= 0 || C <= 0 || FH <= 0 || FW <= 0 || SH <= 0 || SW <= 0 || DH <= 0 ||
        DW <= 0 || PH < 0 || PW < 0)
        return -1;
    s->N = N; s->H = H; s->W = W; s->C = C; s->FH = FH; s->FW = FW;
    s->SH = SH; s->SW = SW; s->DH = DH; s->DW = DW; s->PH = PH; s->PW = PW;
    s->OH = dwo_out_extent(H, FH, SH, DH, PH);
    s->OW = dwo_out_extent(W, FW, SW, DW, PW);
    if (s->OH <= 0 || s->OW <= 0) return -2;
    return 0;
}

/* NHWC / FH x FW x C element offsets. */
#define XIDX(s, n, h, w, c) ((((n) * (s)->H + (h)) * (s)->W + (w)) * (s)->C + (c))
#define YIDX(s, n, h, w, c) ((((n) * (s)->OH + (h)) * (s)->OW + (w)) * (s)->C + (c))
#define WIDX(s, fh, fw, c) ((((fh) * (s)->FW) + (fw)) * (s)->C + (c))

/* ---- threading: one job per channel range ------------------------------ */

typedef struct {
    const dwo_shape *s;
    long c0, c1;
    int kind;               /* 0 fwd, 1 dgrad, 2 wgrad */
    int integer;            /* 0: double, 1: int64 */
    const void *a, *b, *bias;
    void *out, *mag;
} dwo_job;

static double dabs(double v) { return v < 0 ? -v : v; }
static int64_t iabs64(int64_t v) { return v < 0 ? -v : v; }

/* Forward, float64: for every output element, bias then taps fh-major. */
static void fwd_f64(const dwo_job *j) {
    const dwo_shape *s = j->s;
    const double *x = (const double *)j->a, *w = (const double *)j->b;
    const double *bias = (const double *)j->bias;
    double *y = (double *)j->out, *mag = (double *)j->mag;
    long nc = j->c1 - j->c0;
    double *acc = (double *)malloc(sizeof(double) * (size_t)nc);
    double *m = (double *)malloc(sizeof(double) * (size_t)nc);
    for (long n = 0; n < s->N; ++n)
        for (long oh = 0; oh < s->OH; ++oh)
            for (long ow = 0; ow < s->OW; ++ow) {
                for (long c = j->c0; c < j->c1; ++c) {
                    double b = bias ? bias[c] : 0.0;
                    acc[c - j->c0] = b;
                    m[c - j->c0] = dabs(b);
                }
                for (long fh = 0; fh < s->FH; ++fh) {
                    long ih = oh * s->SH - s->PH + fh * s->DH;
                    if (ih < 0 || ih >= s->H) continue;        /* zero padding */
                    for (long fw = 0; fw < s->FW; ++fw) {
                        long iw = ow * s->SW - s->PW + fw * s->DW;
                        if (iw < 0 || iw >= s->W) continue;    /* zero padding */
                        for (long c = j->c0; c < j->c1; ++c) {
                            double p = w[WIDX(s, fh, fw, c)] * x[XIDX(s, n, ih, iw, c)];
                            acc[c - j->c0] += p;
                            m[c - j->c0] += dabs(p);
                        }
                    }
                }
                for (long c = j->c0; c < j->c1; ++c) {
                    y[YIDX(s, n, oh, ow, c)] = acc[c - j->c0];
                    if (mag) mag[YIDX(s, n, oh, ow, c)] = m[c - j->c0];
                }
            }
    free(acc);
    free(m);
}

/* Forward, int64 (int8 data, int32 bias widened by the caller). */
static void fwd_i64(const dwo_job *j) {
    const dwo_shape *s = j->s;
    const int64_t *x = (const int64_t *)j->a, *w = (const int64_t *)j->b;
    const int64_t *bias = (const int64_t *)j->bias;
    int64_t *y = (int64_t *)j->out, *mag = (int64_t *)j->mag;
    for (long n = 0; n < s->N; ++n)
        for (long oh = 0; oh < s->OH; ++oh)
            for (long ow = 0; ow < s->OW; ++ow)
                for (long c = j->c0; c < j->c1; ++c) {
                    int64_t acc = bias ? bias[c] : 0;
                    int64_t m = iabs64(acc);
                    for (long fh = 0; fh < s->FH; ++fh) {
                        long ih = oh * s->SH - s->PH + fh * s->DH;
                        if (ih < 0 || ih >= s->H) continue;
                        for (long fw = 0; fw < s->FW; ++fw) {
                            long iw = ow * s->SW - s->PW + fw * s->DW;
                            if (iw < 0 || iw >= s->W) continue;
                            int64_t p = w[WIDX(s, fh, fw, c)] * x[XIDX(s, n, ih, iw, c)];
                            acc += p;
                            m += iabs64(p);
                        }
                    }
                    y[YIDX(s, n, oh, ow, c)] = acc;
                    if (mag) mag[YIDX(s, n, oh, ow, c)] = m;
                }
}

/* dgrad, float64: scatter every valid tap's product back to its input site. */
static void dgrad_f64(const dwo_job *j) {
    const dwo_shape *s = j->s;
    const double *dy = (const double *)j->a, *w = (const double *)j->b;
    double *dx = (double *)j->out, *mag = (double *)j->mag;
    for (long n = 0; n < s->N; ++n)
        for (long ih = 0; ih < s->H; ++ih)
            for (long iw = 0; iw < s->W; ++iw)
                for (long c = j->c0; c < j->c1; ++c) {
                    dx[XIDX(s, n, ih, iw, c)] = 0.0;
                    if (mag) mag[XIDX(s, n, ih, iw, c)] = 0.0;
                }
    for (long n = 0; n < s->N; ++n)
        for (long oh = 0; oh < s->OH; ++oh)
            for (long ow = 0; ow < s->OW; ++ow)
                for (long fh = 0; fh < s->FH; ++fh) {
                    long ih = oh * s->SH - s->PH + fh * s->DH;
                    if (ih < 0 || ih >= s->H) continue;
                    for (long fw = 0; fw < s->FW; ++fw) {
                        long iw = ow * s->SW - s->PW + fw * s->DW;
                        if (iw < 0 || iw >= s->W) continue;
                        for (long c = j->c0; c < j->c1; ++c) {
                            double p = w[WIDX(s, fh, fw, c)] * dy[YIDX(s, n, oh, ow, c)];
                            dx[XIDX(s, n, ih, iw, c)] += p;
                            if (mag) mag[XIDX(s, n, ih, iw, c)] += dabs(p);
                        }
                    }
                }
}

static void dgrad_i64(const dwo_job *j) {
    const dwo_shape *s = j->s;
    const int64_t *dy = (const int64_t *)j->a, *w = (const int64_t *)j->b;
    int64_t *dx = (int64_t *)j->out, *mag = (int64_t *)j->mag;
    for (long n = 0; n < s->N; ++n)
        for (long ih = 0; ih < s->H; ++ih)
            for (long iw = 0; iw < s->W; ++iw)
                for (long c = j->c0; c < j->c1; ++c) {
                    dx[XIDX(s, n, ih, iw, c)] = 0;
                    if (mag) mag[XIDX(s, n, ih, iw, c)] = 0;
                }
    for (long n = 0; n < s->N; ++n)
        for (long oh = 0; oh < s->OH; ++oh)
            for (long ow = 0; ow < s->OW; ++ow)
                for (long fh = 0; fh < s->FH; ++fh) {
                    long ih = oh * s->SH - s->PH + fh * s->DH;
                    if (ih < 0 || ih >= s->H) continue;
                    for (long fw = 0; fw < s->FW; ++fw) {
                        long iw = ow * s->SW - s->PW + fw * s->DW;
                        if (iw < 0 || iw >= s->W) continue;
                        for (long c = j->c0; c < j->c1; ++c) {
                            int64_t p = w[WIDX(s, fh, fw, c)] * dy[YIDX(s, n, oh, ow, c)];
                            dx[XIDX(s, n, ih, iw, c)] += p;
                            if (mag) mag[XIDX(s, n, ih, iw, c)] += iabs64(p);
                        }
                    }
                }
}

/* wgrad, float64: each filter tap sums dy*x over every output position. */
static void wgrad_f64(const dwo_job *j) {
    const dwo_shape *s = j->s;
    const double *x = (const double *)j->a, *dy = (const double *)j->b;
    double *dw = (double *)j->out, *mag = (double *)j->mag;
    for (long fh = 0; fh < s->FH; ++fh)
        for (long fw = 0; fw < s->FW; ++fw)
            for (long c = j->c0; c < j->c1; ++c) {
                dw[WIDX(s, fh, fw, c)] = 0.0;
                if (mag) mag[WIDX(s, fh, fw, c)] = 0.0;
            }
    for (long n = 0; n < s->N; ++n)
        for (long oh = 0; oh < s->OH; ++oh)
            for (long ow = 0; ow < s->OW; ++ow)
                for (long fh = 0; fh < s->FH; ++fh) {
                    long ih = oh * s->SH - s->PH + fh * s->DH;
                    if (ih < 0 || ih >= s->H) continue;
                    for (long fw = 0; fw < s->FW; ++fw) {
                        long iw = ow * s->SW - s->PW + fw * s->DW;
                        if (iw < 0 || iw >= s->W) continue;
                        for (long c = j->c0; c < j->c1; ++c) {
                            double p = dy[YIDX(s, n, oh, ow, c)] * x[XIDX(s, n, ih, iw, c)];
                            dw[WIDX(s, fh, fw, c)] += p;
                            if (mag) mag[WIDX(s, fh, fw, c)] += dabs(p);
                        }
                    }
                }
}

static void wgrad_i64(const dwo_job *j) {
    const dwo_shape *s = j->s;
    const int64_t *x = (const int64_t *)j->a, *dy = (const int64_t *)j->b;
    int64_t *dw = (int64_t *)j->out, *mag = (int64_t *)j->mag;
    for (long fh = 0; fh < s->FH; ++fh)
        for (long fw = 0; fw < s->FW; ++fw)
            for (long c = j->c0; c < j->c1; ++c) {
                dw[WIDX(s, fh, fw, c)] = 0;
                if (mag) mag[WIDX(s, fh, fw, c)] = 0;
            }
    for (long n = 0; n < s->N; ++n)
        for (long oh = 0; oh < s->OH; ++oh)
            for (long ow = 0; ow < s->OW; ++ow)
                for (long fh = 0; fh < s->FH; ++fh) {
                    long ih = oh * s->SH - s->PH + fh * s->DH;
                    if (ih < 0 || ih >= s->H) continue;
                    for (long fw = 0; fw < s->FW; ++fw) {
                        long iw = ow * s->SW - s->PW + fw * s->DW;
                        if (iw < 0 || iw >= s->W) continue;
                        for (long c = j->c0; c < j->c1; ++c) {
                            int64_t p = dy[YIDX(s, n, oh, ow, c)] * x[XIDX(s, n, ih, iw, c)];
                            dw[WIDX(s, fh, fw, c)] += p;
                            if (mag) mag[WIDX(s, fh, fw, c)] += iabs64(p);
                        }
                    }
                }
}

static void *run_job(void *arg) {
    const dwo_job *j = (const dwo_job *)arg;
    if (j->c0 >= j->c1) return NULL;
    switch (j->kind * 2 + j->integer) {
        case 0: fwd_f64(j); break;
        case 1: fwd_i64(j); break;
        case 2: dgrad_f64(j); break;
        case 3: dgrad_i64(j); break;
        case 4: wgrad_f64(j); break;
        case 5: wgrad_i64(j); break;
        default: break;
    }
    return NULL;
}

static int dispatch(int kind, int integer, long N, long H, long W, long C, long FH, long FW,
                    long SH, long SW, long DH, long DW, long PH, long PW, const void *a, const void *b,
                    const void *bias,
                    void *out, void *mag, int nthreads) {
    dwo_shape s;
    int rc = make_shape(&s, N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW);
    if (rc != 0) return rc;
    if (!a || !b || !out) return -3;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > C) nthreads = (int)C;
    dwo_job *jobs = (dwo_job *)calloc((size_t)nthreads, sizeof(dwo_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return -4; }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].s = &s;
        jobs[t].c0 = C * t / nthreads;
        jobs[t].c1 = C * (t + 1) / nthreads;
        jobs[t].kind = kind;
        jobs[t].integer = integer;
        jobs[t].a = a; jobs[t].b = b; jobs[t].bias = bias;
        jobs[t].out = out; jobs[t].mag = mag;
    }
    char *joined = (char *)calloc((size_t)nthreads, 1);
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, run_job, &jobs[t]) != 0) {
            run_job(&jobs[t]);      /* could not start a thread: do it here */
            joined[t] = 1;
        }
    }
    run_job(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (!joined[t]) pthread_join(tid[t], NULL);
    free(joined);
    free(jobs);
    free(tid);
    return 0;
}

/* ---- exported entry points (return 0 on success, <0 on bad arguments) --- */

int dwo_fwd_f64(long N, long H, long W, long C, long FH, long FW, long SH, long SW, long DH,
                long DW, long PH, long PW,
                const double *x, const double *w, const double *bias, double *y, double *mag,
                int nthreads) {
    return dispatch(0, 0, N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW, x, w, bias, y, mag, nthreads);
}

int dwo_fwd_i64(long N, long H, long W, long C, long FH, long FW, long SH, long SW, long DH,
                long DW, long PH, long PW,
                const int64_t *x, const int64_t *w, const int64_t *bias, int64_t *y,
                int64_t *mag, int nthreads) {
    return dispatch(0, 1, N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW, x, w, bias, y, mag, nthreads);
}

int dwo_dgrad_f64(long N, long H, long W, long C, long FH, long FW, long SH, long SW, long DH,
                long DW, long PH, long PW,
                  const double *dy, const double *w, double *dx, double *mag, int nthreads) {
    return dispatch(1, 0, N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW, dy, w, NULL, dx, mag, nthreads);
}

int dwo_dgrad_i64(long N, long H, long W, long C, long FH, long FW, long SH, long SW, long DH,
                long DW, long PH, long PW,
                  const int64_t *dy, const int64_t *w, int64_t *dx, int64_t *mag, int nthreads) {
    return dispatch(1, 1, N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW, dy, w, NULL, dx, mag, nthreads);
}

int dwo_wgrad_f64(long N, long H, long W, long C, long FH, long FW, long SH, long SW, long DH,
                long DW, long PH, long PW,
                  const double *x, const double *dy, double *dw, double *mag, int nthreads) {
    return dispatch(2, 0, N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW, x, dy, NULL, dw, mag, nthreads);
}

int dwo_wgrad_i64(long N, long H, long W, long C, long FH, long FW, long SH, long SW, long DH,
                long DW, long PH, long PW,
                  const int64_t *x, const int64_t *dy, int64_t *dw, int64_t *mag, int nthreads) {
    return dispatch(2, 1, N, H, W, C, FH, FW, SH, SW, DH, DW, PH, PW, x, dy, NULL, dw, mag, nthreads);
}
