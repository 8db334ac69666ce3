/*
 * oracle.c — plain, slow, fp64 CPU oracle for the forward and backward
 * (vector-Jacobian product) of the weighted sum and of the scaled SiLU.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library.  It shares no code, header,
 * table or constant with the CUDA library; neither includes the other.
 *
 * Sources (web pages, cited by title and section):
 *  [WS]   "Writing Triton Kernels with Autograd: A Minimal End-to-End
 *          Example", §1 Problem Setup (y = x.dot(w), x [N,D], w [D], y [N];
 *          the PyTorch form (x * w).sum(-1)), §3 Backward: Deriving Gradients
 *          First (grad_x = grad_out[:,None] * w[None,:],
 *          grad_w = (x * grad_out[:,None]).sum(0); the two-stage grad_w with
 *          one partial row per BLOCK_N-row tile, then a sum over tiles).
 *  [SILU] "Backward in Triton — autograd.Function and the backward grid",
 *          § A complete minimal example — fused scaled-SiLU (y = w·x·sigmoid(x)
 *          with scalar w; s = sigmoid(x), silu = x·s;
 *          dy/dx = w·(s + silu·(1 − s)); dx = dy·dy/dx; dw = Σ dy·silu).
 *
 * Arithmetic.  Every input is converted exactly to double.  Products of a
 * binary16/bfloat16/binary32 value with a binary32 value are exact in double.
 * Reductions use pairwise summation (N. Higham, Accuracy and Stability of
 * Numerical Algorithms, 2nd ed., §4.2): a range of more than eight terms is
 * split at its midpoint and the two halves' sums are added; up to eight
 * terms are added left to right.  Elementwise results are rounded once, to
 * nearest-even, to the output type.
 *
 * Storage types: 0 = binary32, 1 = binary16, 2 = bfloat16 (raw 16-bit
 * patterns for the last two).
 *
 * Threads.  Built with OpenMP, independent rows (or elements) are computed in
 * parallel, and the upper levels of the long pairwise sums run as separate
 * tasks with the same split points; every result is the same bits at any
 * thread count (orc_set_threads chooses it; tested).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2

/* ------------------------------------------------------------------ */
/* Exact decoding of the storage types.                                */
/* ------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h) {
    const int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);           /* zero or subnormal: m · 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) · 2^(e-15) */
    return s ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 pattern. */
double orc_bf16_to_f64(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* The two 16-bit decodings, tabulated once (65,536 entries each) so that
 * the full-size checks are not dominated by ldexp calls. */
static double* tab_f16 = NULL;
static double* tab_bf16 = NULL;

static void make_tables(void) {
    if (tab_f16) return;
    double* a = (double*)malloc(sizeof(double) * 65536);
    double* b = (double*)malloc(sizeof(double) * 65536);
    for (uint32_t h = 0; h < 65536; h++) {
        a[h] = orc_f16_to_f64((uint16_t)h);
        b[h] = orc_bf16_to_f64((uint16_t)h);
    }
    tab_bf16 = b;
    tab_f16 = a;
}

static double decode(const void* p, int64_t k, int dt) {
    if (dt == ORC_F32) return (double)((const float*)p)[k];
    if (dt == ORC_F16) return tab_f16[((const uint16_t*)p)[k]];
    return tab_bf16[((const uint16_t*)p)[k]];
}

/* ------------------------------------------------------------------ */
/* Rounding to the storage types, to nearest with ties to even.        */
/* The value is scaled by its quantum (a power of two, so exactly),    */
/* rounded to an integer with rint() (the default rounding mode is     */
/* nearest-even), and re-encoded.                                      */
/* ------------------------------------------------------------------ */

/* Generic: p = fraction bits, emin = smallest normal exponent,
 * emax = largest exponent; returns the value after rounding (±inf on
 * overflow). */
static double round_value(double v, int p, int emin, int emax) {
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    const double a = fabs(v);
    int e;
    frexp(a, &e);   /* a = f · 2^e with f in [0.5, 1): exponent of a is e - 1 */
    e -= 1;
    if (e < emin) e = emin;                 /* subnormal quantum */
    const double q = ldexp(1.0, e - p);     /* quantum at this exponent */
    double r = rint(a / q) * q;             /* exact: a/q has at most 53 bits */
    const double maxv = ldexp(2.0 - ldexp(1.0, -p), emax);
    if (r > maxv) r = INFINITY;
    return v < 0 ? -r : r;
}

static uint16_t encode_bits(double r, int p, int emin, int ebits) {
    uint16_t s = signbit(r) ? (uint16_t)(1u << (p + ebits)) : 0;
    if (isnan(r)) return s | (uint16_t)(((1u << ebits) - 1) << p) | (uint16_t)(1u << (p - 1));
    const double a = fabs(r);
    if (isinf(a)) return s | (uint16_t)(((1u << ebits) - 1) << p);
    if (a == 0.0) return s;
    if (a < ldexp(1.0, emin)) /* subnormal: a = m · 2^(emin - p) */
        return s | (uint16_t)(a / ldexp(1.0, emin - p));
    int e;
    const double f = frexp(a, &e); /* a = f·2^e, f in [0.5,1) */
    const int E = e - 1 + ((1 << (ebits - 1)) - 1);
    const uint16_t m = (uint16_t)((f * 2.0 - 1.0) * ldexp(1.0, p));
    return s | (uint16_t)(E << p) | m;
}

uint16_t orc_f64_to_f16(double v) {
    return encode_bits(round_value(v, 10, -14, 15), 10, -14, 5);
}

uint16_t orc_f64_to_bf16(double v) {
    return encode_bits(round_value(v, 7, -126, 127), 7, -126, 8);
}

/* Round to the storage type and write element k of out. */
static void store(void* out, int64_t k, int dt, double v) {
    if (dt == ORC_F32)
        ((float*)out)[k] = (float)v; /* C conversion: IEEE round-to-nearest-even */
    else if (dt == ORC_F16)
        ((uint16_t*)out)[k] = orc_f64_to_f16(v);
    else
        ((uint16_t*)out)[k] = orc_f64_to_bf16(v);
}

/* ------------------------------------------------------------------ */
/* Pairwise summation (Higham §4.2).                                   */
/* ------------------------------------------------------------------ */

double orc_pairwise_sum(const double* t, int64_t n) {
    if (n <= 8) {
        double s = 0.0;
        for (int64_t i = 0; i < n; i++) s += t[i];
        return s;
    }
    const int64_t h = n / 2;
    return orc_pairwise_sum(t, h) + orc_pairwise_sum(t + h, n - h);
}

/* ------------------------------------------------------------------ */
/* Threads.                                                            */
/* ------------------------------------------------------------------ */

/* Sets the number of threads (n >= 1) and returns the previous number; a
 * build without OpenMP has one thread and ignores n. */
int orc_set_threads(int n) {
#ifdef _OPENMP
    const int old = omp_get_max_threads();
    if (n >= 1) omp_set_num_threads(n);
    return old;
#else
    (void)n;
    return 1;
#endif
}

static int n_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int thread_id(void) {
#ifdef _OPENMP
    return omp_get_thread_num();
#else
    return 0;
#endif
}

static void set_flag(int* f) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
    *f = 1;
}

/* A sub-range shorter than this many terms is summed by one thread. */
#define TASK_MIN_TERMS ((int64_t)1 << 16)

/* orc_pairwise_sum with the two halves of each range longer than
 * TASK_MIN_TERMS summed as separate tasks: the same tree. */
static double pairwise_task(const double* t, int64_t n) {
    if (n <= TASK_MIN_TERMS) return orc_pairwise_sum(t, n);
    const int64_t h = n / 2;
    double left = 0.0, right = 0.0;
#ifdef _OPENMP
#pragma omp task shared(left) firstprivate(t, h)
#endif
    left = pairwise_task(t, h);
    right = pairwise_task(t + h, n - h);
#ifdef _OPENMP
#pragma omp taskwait
#endif
    return left + right;
}

static double pairwise_par(const double* t, int64_t n) {
    double s = 0.0;
#ifdef _OPENMP
#pragma omp parallel
#pragma omp single
#endif
    s = pairwise_task(t, n);
    return s;
}

/* ------------------------------------------------------------------ */
/* Weighted sum, forward  [WS §1, §2]:  y[i] = Σ_d x[i,d] · w[d].      */
/* ------------------------------------------------------------------ */

/* x: [N, D] storage type dt with row stride ldx (elements); w: [D] binary32.
 * Outputs (any may be NULL): y_exact[i] the fp64 pairwise sum,
 * y_abs[i] = Σ_d |x[i,d]·w[d]|, y_out[i] = y_exact[i] rounded to dt. */
int orc_ws_fwd(const void* x, int64_t ldx, const float* w, int64_t N, int64_t D, int dt,
               double* y_exact, double* y_abs, void* y_out) {
    if (!x || !w || N < 0 || D < 0 || ldx < D || dt < 0 || dt > 2) return -1;
    make_tables();
    const int64_t Dm = D > 0 ? D : 1;
    double* tb = (double*)malloc(sizeof(double) * (size_t)Dm * 2 * (size_t)n_threads());
    if (!tb) return -2;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < N; i++) {
        double* t = tb + (size_t)thread_id() * 2 * Dm;  /* this thread's scratch */
        double* ta = t + Dm;
        for (int64_t d = 0; d < D; d++) {
            t[d] = decode(x, i * ldx + d, dt) * (double)w[d];
            ta[d] = fabs(t[d]);
        }
        const double y = orc_pairwise_sum(t, D);
        if (y_exact) y_exact[i] = y;
        if (y_abs) y_abs[i] = orc_pairwise_sum(ta, D);
        if (y_out) store(y_out, i, dt, y);
    }
    free(tb);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Weighted sum, backward  [WS §3, §4]:                                */
/*   dx[i,d]     = dy[i] · w[d]                                        */
/*   grad_w[d]   = Σ_i x[i,d] · dy[i]                                  */
/*   partial[p,d]= Σ_{i in tile p} x[i,d] · dy[i],                      */
/*                 tile p = rows p·block_n .. min(N, (p+1)·block_n) - 1 */
/* ------------------------------------------------------------------ */

/* Column-wise pairwise sums over rows [a, b) of the terms x[i,d]·dy[i]
 * into out[0..D) and of |x[i,d]·dy[i]| into out_abs[0..D) (either may be
 * NULL).  The split points are those of orc_pairwise_sum applied to each
 * column separately; rows are walked in storage order so that the loops
 * read memory sequentially.  scratch holds 2·D doubles per recursion level. */
static void colsum(const void* x, int64_t ldx, const void* dy, int dt, int64_t a, int64_t b,
                   int64_t D, double* out, double* out_abs, double* scratch) {
    const int64_t n = b - a;
    if (n <= 8) {
        for (int64_t d = 0; d < D; d++) {
            if (out) out[d] = 0.0;
            if (out_abs) out_abs[d] = 0.0;
        }
        for (int64_t i = a; i < b; i++) {
            const double g = decode(dy, i, dt);
            for (int64_t d = 0; d < D; d++) {
                const double term = decode(x, i * ldx + d, dt) * g;
                if (out) out[d] += term;
                if (out_abs) out_abs[d] += fabs(term);
            }
        }
        return;
    }
    const int64_t h = n / 2;
    double* r = scratch;          /* right half, signed */
    double* ra = scratch + D;     /* right half, absolute */
    colsum(x, ldx, dy, dt, a, a + h, D, out, out_abs, scratch + 2 * D);
    colsum(x, ldx, dy, dt, a + h, b, D, out ? r : NULL, out_abs ? ra : NULL, scratch + 2 * D);
    for (int64_t d = 0; d < D; d++) {
        if (out) out[d] += r[d];
        if (out_abs) out_abs[d] += ra[d];
    }
}

/* colsum with the upper levels of the recursion (ranges of more than
 * TASK_MIN_TERMS terms) run as tasks: the same split points and the same
 * additions, so the same result at any thread count. */
static void colsum_task(const void* x, int64_t ldx, const void* dy, int dt, int64_t a, int64_t b,
                        int64_t D, double* out, double* out_abs, int* err) {
    const int64_t n = b - a;
    const int64_t Dm = D > 0 ? D : 1;
    if (n <= 8 || n * Dm <= TASK_MIN_TERMS) {
        /* recursion depth <= 64; each level needs 2·D doubles */
        double* scratch = (double*)malloc(sizeof(double) * (size_t)Dm * 2 * 66);
        if (!scratch) { set_flag(err); return; }
        colsum(x, ldx, dy, dt, a, b, D, out, out_abs, scratch);
        free(scratch);
        return;
    }
    const int64_t h = n / 2;
    double* r = (double*)malloc(sizeof(double) * (size_t)Dm * 2);  /* right half */
    if (!r) { set_flag(err); return; }
    double* ra = r + Dm;
#ifdef _OPENMP
#pragma omp task firstprivate(x, ldx, dy, dt, a, h, D, out, out_abs, err)
#endif
    colsum_task(x, ldx, dy, dt, a, a + h, D, out, out_abs, err);
    colsum_task(x, ldx, dy, dt, a + h, b, D, out ? r : NULL, out_abs ? ra : NULL, err);
#ifdef _OPENMP
#pragma omp taskwait
#endif
    for (int64_t d = 0; d < D; d++) {
        if (out) out[d] += r[d];
        if (out_abs) out_abs[d] += ra[d];
    }
    free(r);
}

static int colsum_range(const void* x, int64_t ldx, const void* dy, int dt, int64_t a, int64_t b,
                        int64_t D, double* out, double* out_abs) {
    int err = 0;
#ifdef _OPENMP
#pragma omp parallel
#pragma omp single
#endif
    colsum_task(x, ldx, dy, dt, a, b, D, out, out_abs, &err);
    return err ? -2 : 0;
}

/* Inputs: x [N,D] (row stride ldx), w [D] binary32, dy [N], storage dt.
 * Outputs (any may be NULL):
 *   dx_out [N,D] contiguous in dt: dy[i]·w[d] (an exact product) rounded once;
 *   grad_w[d], grad_w_abs[d] = Σ_i |x[i,d]·dy[i]|;
 *   partial [ceil(N/block_n), D] (only when block_n > 0). */
int orc_ws_bwd(const void* x, int64_t ldx, const float* w, const void* dy, int64_t N, int64_t D,
               int dt, void* dx_out, double* grad_w, double* grad_w_abs, int64_t block_n,
               double* partial) {
    if (!x || !w || !dy || N < 0 || D < 0 || ldx < D || dt < 0 || dt > 2) return -1;
    make_tables();
    if (dx_out) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t i = 0; i < N; i++) {
            const double g = decode(dy, i, dt);
            for (int64_t d = 0; d < D; d++) store(dx_out, i * D + d, dt, g * (double)w[d]);
        }
    }
    if ((grad_w || grad_w_abs) && colsum_range(x, ldx, dy, dt, 0, N, D, grad_w, grad_w_abs))
        return -2;
    if (partial && block_n > 0) {
        const int64_t P = (N + block_n - 1) / block_n;
        for (int64_t p = 0; p < P; p++) {
            const int64_t a = p * block_n, b = (a + block_n < N) ? a + block_n : N;
            if (colsum_range(x, ldx, dy, dt, a, b, D, partial + p * D, NULL)) return -2;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Scaled SiLU  [SILU]:                                                */
/*   s = 1 / (1 + exp(-x)),  y = w·x·s                                  */
/*   dy/dx = w·(s + x·s·(1 - s)),  dx = dy · dy/dx                      */
/*   dw = Σ_k dy_k · x_k · s_k                                          */
/* ------------------------------------------------------------------ */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* x [n] in dt, scalar w.  Outputs (any may be NULL): y_exact, y_out (dt). */
int orc_silu_fwd(const void* x, double w, int64_t n, int dt, double* y_exact, void* y_out) {
    if (!x || n < 0 || dt < 0 || dt > 2) return -1;
    make_tables();
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t k = 0; k < n; k++) {
        const double xv = decode(x, k, dt);
        const double y = w * xv * sigmoid(xv);
        if (y_exact) y_exact[k] = y;
        if (y_out) store(y_out, k, dt, y);
    }
    return 0;
}

/* dy, x [n] in dt, scalar w.  Outputs (any may be NULL):
 *   dx_exact[k], dx_scale[k] = |dy·w|·(s + |x·s·(1 - s)|) (the sum of the
 *   magnitudes of the two terms of dy/dx, scaled), dx_out[k] (dt),
 *   dw = Σ dy·x·s (pairwise), dw_abs = Σ |dy·x·s|. */
int orc_silu_bwd(const void* dy, const void* x, double w, int64_t n, int dt, double* dx_exact,
                 double* dx_scale, void* dx_out, double* dw, double* dw_abs) {
    if (!dy || !x || n < 0 || dt < 0 || dt > 2) return -1;
    make_tables();
    double* t = NULL;
    double* ta = NULL;
    if (dw || dw_abs) {
        t = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        ta = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        if (!t || !ta) { free(t); free(ta); return -2; }
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t k = 0; k < n; k++) {
        const double g = decode(dy, k, dt);
        const double xv = decode(x, k, dt);
        const double s = sigmoid(xv);
        const double silu = xv * s;
        const double dydx = w * (s + silu * (1.0 - s));
        const double dx = g * dydx;
        if (dx_exact) dx_exact[k] = dx;
        if (dx_scale) dx_scale[k] = fabs(g * w) * (s + fabs(silu * (1.0 - s)));
        if (dx_out) store(dx_out, k, dt, dx);
        if (t) {
            t[k] = g * silu;
            ta[k] = fabs(t[k]);
        }
    }
    if (dw) *dw = pairwise_par(t, n);
    if (dw_abs) *dw_abs = pairwise_par(ta, n);
    free(t);
    free(ta);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Softmax over rows  ["Backprop for kernel writers", §04 The duality:  */
/* softmax backward collapses the dense Jacobian to one row scalar]:    */
/*   y[i,j]  = exp(x[i,j] - m_i) / Σ_k exp(x[i,k] - m_i),  m_i = max_k x */
/*   dx[i,j] = y[i,j] · (dy[i,j] - s_i),  s_i = Σ_k dy[i,k] · y[i,k]     */
/* ------------------------------------------------------------------ */

/* x [N, D] (row stride ldx), storage dt.  Outputs (any may be NULL):
 * y_exact [N*D] contiguous fp64, y_out [N, D] contiguous in dt. */
int orc_softmax_fwd(const void* x, int64_t ldx, int64_t N, int64_t D, int dt, double* y_exact,
                    void* y_out) {
    if (!x || N < 0 || D < 0 || ldx < D || dt < 0 || dt > 2) return -1;
    make_tables();
    const int64_t Dm = D > 0 ? D : 1;
    double* eb = (double*)malloc(sizeof(double) * (size_t)Dm * (size_t)n_threads());
    if (!eb) return -2;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < N; i++) {
        double* e = eb + (size_t)thread_id() * Dm;  /* this thread's scratch */
        double m = -INFINITY;
        for (int64_t j = 0; j < D; j++) {
            const double v = decode(x, i * ldx + j, dt);
            if (v > m) m = v;
        }
        for (int64_t j = 0; j < D; j++) e[j] = exp(decode(x, i * ldx + j, dt) - m);
        const double S = orc_pairwise_sum(e, D);
        for (int64_t j = 0; j < D; j++) {
            const double y = e[j] / S;
            if (y_exact) y_exact[i * D + j] = y;
            if (y_out) store(y_out, i * D + j, dt, y);
        }
    }
    free(eb);
    return 0;
}

/* y, dy [N, D] contiguous in dt (y is the forward's stored output).
 * Outputs (any may be NULL): dx_exact, dx_scale = |y|·(|dy| + Σ_k |dy_k·y_k|)
 * (the magnitude of the two cancelling terms), dx_out (dt), s_exact [N]. */
int orc_softmax_bwd(const void* y, const void* dy, int64_t N, int64_t D, int dt, double* dx_exact,
                    double* dx_scale, void* dx_out, double* s_exact) {
    if (!y || !dy || N < 0 || D < 0 || dt < 0 || dt > 2) return -1;
    make_tables();
    const int64_t Dm = D > 0 ? D : 1;
    double* tb = (double*)malloc(sizeof(double) * (size_t)Dm * 2 * (size_t)n_threads());
    if (!tb) return -2;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < N; i++) {
        double* t = tb + (size_t)thread_id() * 2 * Dm;  /* this thread's scratch */
        double* ta = t + Dm;
        for (int64_t j = 0; j < D; j++) {
            t[j] = decode(dy, i * D + j, dt) * decode(y, i * D + j, dt);
            ta[j] = fabs(t[j]);
        }
        const double s = orc_pairwise_sum(t, D);
        const double sa = orc_pairwise_sum(ta, D);
        if (s_exact) s_exact[i] = s;
        for (int64_t j = 0; j < D; j++) {
            const double yv = decode(y, i * D + j, dt), g = decode(dy, i * D + j, dt);
            const double dx = yv * (g - s);
            if (dx_exact) dx_exact[i * D + j] = dx;
            if (dx_scale) dx_scale[i * D + j] = fabs(yv) * (fabs(g) + sa);
            if (dx_out) store(dx_out, i * D + j, dt, dx);
        }
    }
    free(tb);
    return 0;
}

/* ------------------------------------------------------------------ */
/* RMSNorm and LayerNorm over rows, with their backward.  The pages     */
/* name both ("Backward in Triton", § Save vs recompute: the RMSNorm    */
/* rstd recompute; § The backward grid ...: RMSNorm's dw sums a length-d */
/* partial from every row; "Backprop for kernel writers", §04: LayerNorm */
/* collapses to two row scalars plus batch-axis parameter gradients)    */
/* but print no formulas; these are the textbook definitions.          */
/*   RMSNorm:   r = 1/sqrt(mean_j x_j^2 + eps),  y = x·r·w              */
/*              xh = x·r, g = dy·w,                                      */
/*              dx = r·(g − xh·mean_j(g·xh)),  dw = Σ_i dy·xh            */
/*   LayerNorm: mu = mean x, r = 1/sqrt(mean (x−mu)^2 + eps),            */
/*              xh = (x−mu)·r, y = xh·w + b,                             */
/*              dx = r·(g − mean g − xh·mean(g·xh)),                     */
/*              dw = Σ_i dy·xh,  db = Σ_i dy                             */
/* ------------------------------------------------------------------ */

/* Row statistics: mean (LayerNorm only) and r, both from pairwise sums. */
static void norm_stats(const void* x, int64_t off, int64_t D, int dt, int ln, double eps,
                       double* t, double* mu_out, double* r_out) {
    double mu = 0.0;
    if (ln) {
        for (int64_t j = 0; j < D; j++) t[j] = decode(x, off + j, dt);
        mu = orc_pairwise_sum(t, D) / (double)D;
    }
    for (int64_t j = 0; j < D; j++) {
        const double c = decode(x, off + j, dt) - mu;
        t[j] = c * c;
    }
    *mu_out = mu;
    *r_out = 1.0 / sqrt(orc_pairwise_sum(t, D) / (double)D + eps);
}

/* x [N, D] (row stride ldx), w, b [D] binary32 (b unused unless ln).
 * Outputs (any may be NULL): y_exact [N*D], y_scale [N*D] (magnitude of the
 * terms: (|x| + |mu|)·r·|w| + |b|), y_out (dt, contiguous), r_out [N], mu_out [N]. */
int orc_norm_fwd(const void* x, int64_t ldx, const float* w, const float* b, double eps, int ln,
                 int64_t N, int64_t D, int dt, double* y_exact, double* y_scale, void* y_out,
                 double* r_out, double* mu_out) {
    if (!x || !w || (ln && !b) || N < 0 || D <= 0 || ldx < D || dt < 0 || dt > 2) return -1;
    make_tables();
    double* tb = (double*)malloc(sizeof(double) * (size_t)D * (size_t)n_threads());
    if (!tb) return -2;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < N; i++) {
        double* t = tb + (size_t)thread_id() * D;  /* this thread's scratch */
        double mu, r;
        norm_stats(x, i * ldx, D, dt, ln, eps, t, &mu, &r);
        if (r_out) r_out[i] = r;
        if (mu_out) mu_out[i] = mu;
        for (int64_t j = 0; j < D; j++) {
            const double xv = decode(x, i * ldx + j, dt);
            const double y = (xv - mu) * r * (double)w[j] + (ln ? (double)b[j] : 0.0);
            if (y_exact) y_exact[i * D + j] = y;
            if (y_scale)
                y_scale[i * D + j] = (fabs(xv) + fabs(mu)) * r * fabs((double)w[j]) +
                                     (ln ? fabs((double)b[j]) : 0.0);
            if (y_out) store(y_out, i * D + j, dt, y);
        }
    }
    free(tb);
    return 0;
}

/* Column-wise pairwise sums over rows [a, b) of dy[i,j]·xh[i,j] (into
 * gw/gwa, signed and absolute) and dy[i,j] (into gb/gba), xh = (x − mu_i)·r_i,
 * with the split points of orc_pairwise_sum; rows walked in storage order.
 * scratch: 4·D doubles per recursion level. */
static void normcol(const void* x, int64_t ldx, const void* dy, int dt, const double* mu,
                    const double* r, int64_t a, int64_t b, int64_t D, double* gw, double* gwa,
                    double* gb, double* gba, double* scratch) {
    const int64_t n = b - a;
    if (n <= 8) {
        for (int64_t j = 0; j < D; j++) gw[j] = gwa[j] = gb[j] = gba[j] = 0.0;
        for (int64_t i = a; i < b; i++)
            for (int64_t j = 0; j < D; j++) {
                const double g = decode(dy, i * D + j, dt);
                const double t = g * ((decode(x, i * ldx + j, dt) - mu[i]) * r[i]);
                gw[j] += t;
                gwa[j] += fabs(t);
                gb[j] += g;
                gba[j] += fabs(g);
            }
        return;
    }
    const int64_t h = n / 2;
    double* rw = scratch;
    double* rwa = scratch + D;
    double* rb = scratch + 2 * D;
    double* rba = scratch + 3 * D;
    normcol(x, ldx, dy, dt, mu, r, a, a + h, D, gw, gwa, gb, gba, scratch + 4 * D);
    normcol(x, ldx, dy, dt, mu, r, a + h, b, D, rw, rwa, rb, rba, scratch + 4 * D);
    for (int64_t j = 0; j < D; j++) {
        gw[j] += rw[j];
        gwa[j] += rwa[j];
        gb[j] += rb[j];
        gba[j] += rba[j];
    }
}

/* normcol with the upper levels of the recursion run as tasks (as
 * colsum_task): the same split points and additions. */
static void normcol_task(const void* x, int64_t ldx, const void* dy, int dt, const double* mu,
                         const double* r, int64_t a, int64_t b, int64_t D, double* gw, double* gwa,
                         double* gb, double* gba, int* err) {
    const int64_t n = b - a;
    if (n <= 8 || n * D <= TASK_MIN_TERMS) {
        double* scratch = (double*)malloc(sizeof(double) * (size_t)D * 4 * 68);
        if (!scratch) { set_flag(err); return; }
        normcol(x, ldx, dy, dt, mu, r, a, b, D, gw, gwa, gb, gba, scratch);
        free(scratch);
        return;
    }
    const int64_t h = n / 2;
    double* rr = (double*)malloc(sizeof(double) * (size_t)D * 4);  /* right half */
    if (!rr) { set_flag(err); return; }
#ifdef _OPENMP
#pragma omp task firstprivate(x, ldx, dy, dt, mu, r, a, h, D, gw, gwa, gb, gba, err)
#endif
    normcol_task(x, ldx, dy, dt, mu, r, a, a + h, D, gw, gwa, gb, gba, err);
    normcol_task(x, ldx, dy, dt, mu, r, a + h, b, D, rr, rr + D, rr + 2 * D, rr + 3 * D, err);
#ifdef _OPENMP
#pragma omp taskwait
#endif
    for (int64_t j = 0; j < D; j++) {
        gw[j] += rr[j];
        gwa[j] += rr[D + j];
        gb[j] += rr[2 * D + j];
        gba[j] += rr[3 * D + j];
    }
    free(rr);
}

/* x [N, D] (row stride ldx), w [D], dy [N, D] contiguous, storage dt.
 * Outputs (any may be NULL): dx_exact, dx_scale (|r|·(|g| + mean|g| + |xh|·mean|g·xh|)),
 * dx_out (dt, contiguous), grad_w / grad_w_abs [D], grad_b / grad_b_abs [D] (ln only). */
int orc_norm_bwd(const void* x, int64_t ldx, const float* w, const void* dy, double eps, int ln,
                 int64_t N, int64_t D, int dt, double* dx_exact, double* dx_scale, void* dx_out,
                 double* grad_w, double* grad_w_abs, double* grad_b, double* grad_b_abs) {
    if (!x || !w || !dy || N < 0 || D <= 0 || ldx < D || dt < 0 || dt > 2) return -1;
    make_tables();
    double* tb = (double*)malloc(sizeof(double) * (size_t)D * 2 * (size_t)n_threads());
    double* mus = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double* rs = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!tb || !mus || !rs) {
        free(tb); free(mus); free(rs);
        return -2;
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < N; i++) {
        double* t = tb + (size_t)thread_id() * 2 * D;  /* this thread's scratch */
        double* t2 = t + D;
        double mu, r;
        norm_stats(x, i * ldx, D, dt, ln, eps, t, &mu, &r);
        mus[i] = mu;
        rs[i] = r;
        if (!dx_exact && !dx_scale && !dx_out) continue;
        /* mean g, mean g·xh (and their magnitudes for the tolerance scale) */
        for (int64_t j = 0; j < D; j++) t[j] = decode(dy, i * D + j, dt) * (double)w[j];
        const double mg = ln ? orc_pairwise_sum(t, D) / (double)D : 0.0;
        for (int64_t j = 0; j < D; j++) t2[j] = fabs(t[j]);
        const double mga = ln ? orc_pairwise_sum(t2, D) / (double)D : 0.0;
        for (int64_t j = 0; j < D; j++) t2[j] = t[j] * ((decode(x, i * ldx + j, dt) - mu) * r);
        const double mgx = orc_pairwise_sum(t2, D) / (double)D;
        for (int64_t j = 0; j < D; j++) t2[j] = fabs(t2[j]);
        const double mgxa = orc_pairwise_sum(t2, D) / (double)D;
        for (int64_t j = 0; j < D; j++) {
            const double xh = (decode(x, i * ldx + j, dt) - mu) * r;
            const double g = t[j];
            const double dx = r * (g - mg - xh * mgx);
            if (dx_exact) dx_exact[i * D + j] = dx;
            if (dx_scale) dx_scale[i * D + j] = fabs(r) * (fabs(g) + mga + fabs(xh) * mgxa);
            if (dx_out) store(dx_out, i * D + j, dt, dx);
        }
    }
    if (grad_w || grad_w_abs || grad_b || grad_b_abs) {
        double* gw = (double*)malloc(sizeof(double) * (size_t)D * 4);
        int err = 0;
        if (gw) {
#ifdef _OPENMP
#pragma omp parallel
#pragma omp single
#endif
            normcol_task(x, ldx, dy, dt, mus, rs, 0, N, D, gw, gw + D, gw + 2 * D, gw + 3 * D, &err);
        }
        if (!gw || err) {
            free(gw); free(tb); free(mus); free(rs);
            return -2;
        }
        for (int64_t j = 0; j < D; j++) {
            if (grad_w) grad_w[j] = gw[j];
            if (grad_w_abs) grad_w_abs[j] = gw[D + j];
            if (ln && grad_b) grad_b[j] = gw[2 * D + j];
            if (ln && grad_b_abs) grad_b_abs[j] = gw[3 * D + j];
        }
        free(gw);
    }
    free(tb); free(mus); free(rs);
    return 0;
}
