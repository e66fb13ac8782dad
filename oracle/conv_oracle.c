/*
 * conv_oracle.c -- the CPU oracle for 2D convolution (fprop, dgrad, wgrad,
 * dense and grouped, 3D, int8 fprop with requantisation, int8 dgrad and
 * wgrad with int32 results) and the
 * NCHW<->NHWC permutes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this code; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no source, header, table or helper with the CUDA path.
 *
 * Every sum is a plain loop over the definition, accumulated in double
 * (int64 for the int8 path).  No blocking, no reordering, no im2col.  Work is
 * split across POSIX threads by output element only; each element is
 * computed by exactly one thread with the same loop order, so results do not
 * depend on the thread count.
 *
 * Layouts (all row-major, innermost last):
 *   X  [N][H][W][C]      activations, NHWC
 *   Wt [K][R][S][C]      filters, KRSC
 *   Y  [N][P][Q][K]      fprop output / dgrad input dY
 *   dX [N][H][W][C]      dgrad output
 *   dW [K][R][S][C]      wgrad output
 *
 * Sources (pages, by title and section):
 *   - output size: CUTLASS Python example "03_basic_conv2d.ipynb", section
 *     "General setup" (cutlass.Conv2d.output_size with padding, stride,
 *     dilation); the dilation-free special case is the formula in
 *     tensorcore "docs/conv2d.md", section "Output spatial dims".
 *   - fprop with alpha/beta: 03_basic_conv2d.ipynb, section "Declaring and
 *     running a Conv2d Fprop" (alpha * conv2d(input, weight) + beta * C).
 *   - bias: tensorcore docs/conv2d.md, section "Strategy" (Y += bias,
 *     optional, one value per output channel).
 *   - ReLU after the bias add: PyTorch quantized cuDNN Conv.cpp,
 *     apply_impl_helper<kReluFused> (relu applied to conv + bias).
 *   - dgrad / wgrad with alpha/beta: 03_basic_conv2d.ipynb, section
 *     "Declaring and running Conv2d Dgrad and Wgrad" (the gradients of
 *     conv2d with respect to its input and its weight).
 *   - wgrad as a sum over images of per-image products: tensorcore
 *     docs/conv2d.md, section "Strategy", dWeight.
 *   - int8: apply_impl_helper<kReluFused>: requantize multiplier
 *     act_scale * weight_scale / output_scale computed in double, applied to
 *     relu(conv + bias) and stored as int8.
 *
 * Readings where the pages leave a step open (each one is also listed in the
 * design notes): fp64 / int64 accumulation stands for "exact"; the output
 * conversion to fp16/bf16 is round-to-nearest-even; beta == 0 means C is not
 * read; the int8 bias is int32 in accumulator units; int8 rounding is
 * half-to-even with saturation to [-128, 127]; the multiplier is the fp32
 * value of the double quotient.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int N, H, W, C, K, R, S;
    int pad_h, pad_w, stride_h, stride_w, dil_h, dil_w;
} oracle_problem;

/* ------------------------------------------------------------------------ */
/* Output size                                                               */
/* ------------------------------------------------------------------------ */

/* out = floor((in + 2*pad - dil*(k-1) - 1) / stride) + 1.  Returns a value
 * <= 0 when no output position exists (the caller treats that as invalid). */
int oracle_out_size(int in, int pad, int dil, int k, int stride)
{
    long long span = (long long)in + 2LL * pad - (long long)dil * (k - 1) - 1;
    if (span < 0) return 0;
    return (int)(span / stride) + 1;
}

/* ------------------------------------------------------------------------ */
/* Threading: split [0, count) into contiguous chunks, one per thread.       */
/* ------------------------------------------------------------------------ */

typedef void (*oracle_elem_fn)(const void *ctx, int64_t j);

typedef struct {
    oracle_elem_fn fn;
    const void *ctx;
    int64_t begin, end;
} oracle_chunk;

static void *oracle_run_chunk(void *arg)
{
    oracle_chunk *c = (oracle_chunk *)arg;
    for (int64_t j = c->begin; j < c->end; ++j) c->fn(c->ctx, j);
    return NULL;
}

static void oracle_parallel(oracle_elem_fn fn, const void *ctx, int64_t count, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > count) nthreads = (int)(count > 0 ? count : 1);
    pthread_t tid[256];
    int created[256];
    oracle_chunk chunk[256];
    for (int t = 0; t < nthreads; ++t) {
        chunk[t].fn = fn;
        chunk[t].ctx = ctx;
        chunk[t].begin = count * t / nthreads;
        chunk[t].end = count * (t + 1) / nthreads;
        created[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        created[t] = pthread_create(&tid[t], NULL, oracle_run_chunk, &chunk[t]) == 0;
    oracle_run_chunk(&chunk[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (created[t]) pthread_join(tid[t], NULL);
        else oracle_run_chunk(&chunk[t]); /* no thread could start: run it here */
    }
}

/* ------------------------------------------------------------------------ */
/* fprop                                                                     */
/*   Y[n,p,q,k] = relu?( alpha * sum_{r,s,c} X[n, p*sh - ph + r*dh,          */
/*                          q*sw - pw + s*dw, c] * W[k,r,s,c]                */
/*                       + beta * Cin[n,p,q,k] + bias[k] )                   */
/* Out-of-range input positions contribute nothing (zero padding).           */
/* ------------------------------------------------------------------------ */

typedef struct {
    oracle_problem pb;
    int P, Q;
    const double *X, *Wt, *bias, *Cin;
    double alpha, beta;
    int relu;
    const int64_t *idx;
    double *Y, *A;
} fprop_ctx;

static void fprop_elem(const void *vctx, int64_t j)
{
    const fprop_ctx *t = (const fprop_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int k = (int)(rem % p->K); rem /= p->K;
    int q = (int)(rem % t->Q); rem /= t->Q;
    int pp = (int)(rem % t->P); rem /= t->P;
    int n = (int)rem;
    double sum = 0.0, asum = 0.0;
    for (int r = 0; r < p->R; ++r) {
        int h = pp * p->stride_h - p->pad_h + r * p->dil_h;
        if (h < 0 || h >= p->H) continue;
        for (int s = 0; s < p->S; ++s) {
            int w = q * p->stride_w - p->pad_w + s * p->dil_w;
            if (w < 0 || w >= p->W) continue;
            for (int c = 0; c < p->C; ++c) {
                double x = t->X[(((int64_t)n * p->H + h) * p->W + w) * p->C + c];
                double f = t->Wt[(((int64_t)k * p->R + r) * p->S + s) * p->C + c];
                sum += x * f;
                asum += fabs(x * f);
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    if (t->bias) v += t->bias[k];
    if (t->relu && v < 0.0) v = 0.0;
    t->Y[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

/* idx: optional list of linear output indices (into [N][P][Q][K]); when NULL
 * every output is computed and count must equal N*P*Q*K.  Y[j] and A[j]
 * receive the value and sum |x*w| of element idx[j] (or j).  A may be NULL.
 * Returns 0, or -1 if the output size is empty. */
int oracle_fprop(const oracle_problem *pb, const double *X, const double *Wt,
                 const double *bias, const double *Cin, double alpha, double beta,
                 int relu, const int64_t *idx, int64_t count, double *Y, double *A,
                 int nthreads)
{
    fprop_ctx t;
    t.pb = *pb;
    t.P = oracle_out_size(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
    t.Q = oracle_out_size(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
    if (t.P <= 0 || t.Q <= 0) return -1;
    t.X = X; t.Wt = Wt; t.bias = bias; t.Cin = Cin;
    t.alpha = alpha; t.beta = beta; t.relu = relu;
    t.idx = idx; t.Y = Y; t.A = A;
    oracle_parallel(fprop_elem, &t, count, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* dgrad: the gradient of fprop with respect to X.                           */
/*   dX[n,h,w,c] = alpha * sum over (k, r, s) and the output position (p, q) */
/*   that reads X[n,h,w,c] through tap (r, s), i.e. p*sh - ph + r*dh == h    */
/*   and q*sw - pw + s*dw == w with 0 <= p < P, 0 <= q < Q, of               */
/*   dY[n,p,q,k] * W[k,r,s,c];  plus beta * Cin[n,h,w,c].                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    oracle_problem pb;
    int P, Q;
    const double *dY, *Wt, *Cin;
    double alpha, beta;
    const int64_t *idx;
    double *dX, *A;
} dgrad_ctx;

static void dgrad_elem(const void *vctx, int64_t j)
{
    const dgrad_ctx *t = (const dgrad_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int c = (int)(rem % p->C); rem /= p->C;
    int w = (int)(rem % p->W); rem /= p->W;
    int h = (int)(rem % p->H); rem /= p->H;
    int n = (int)rem;
    double sum = 0.0, asum = 0.0;
    for (int r = 0; r < p->R; ++r) {
        int th = h + p->pad_h - r * p->dil_h;      /* = pp * stride_h */
        if (th < 0 || th % p->stride_h != 0) continue;
        int pp = th / p->stride_h;
        if (pp >= t->P) continue;
        for (int s = 0; s < p->S; ++s) {
            int tw = w + p->pad_w - s * p->dil_w;  /* = q * stride_w */
            if (tw < 0 || tw % p->stride_w != 0) continue;
            int q = tw / p->stride_w;
            if (q >= t->Q) continue;
            for (int k = 0; k < p->K; ++k) {
                double g = t->dY[(((int64_t)n * t->P + pp) * t->Q + q) * p->K + k];
                double f = t->Wt[(((int64_t)k * p->R + r) * p->S + s) * p->C + c];
                sum += g * f;
                asum += fabs(g * f);
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    t->dX[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

/* idx indexes [N][H][W][C]. */
int oracle_dgrad(const oracle_problem *pb, const double *dY, const double *Wt,
                 const double *Cin, double alpha, double beta, const int64_t *idx,
                 int64_t count, double *dX, double *A, int nthreads)
{
    dgrad_ctx t;
    t.pb = *pb;
    t.P = oracle_out_size(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
    t.Q = oracle_out_size(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
    if (t.P <= 0 || t.Q <= 0) return -1;
    t.dY = dY; t.Wt = Wt; t.Cin = Cin;
    t.alpha = alpha; t.beta = beta;
    t.idx = idx; t.dX = dX; t.A = A;
    oracle_parallel(dgrad_elem, &t, count, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* wgrad: the gradient of fprop with respect to W.                           */
/*   dW[k,r,s,c] = alpha * sum_{n,p,q} dY[n,p,q,k] *                          */
/*                 X[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c]               */
/*                 + beta * Cin[k,r,s,c]                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    oracle_problem pb;
    int P, Q;
    const double *X, *dY, *Cin;
    double alpha, beta;
    const int64_t *idx;
    double *dW, *A;
} wgrad_ctx;

static void wgrad_elem(const void *vctx, int64_t j)
{
    const wgrad_ctx *t = (const wgrad_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int c = (int)(rem % p->C); rem /= p->C;
    int s = (int)(rem % p->S); rem /= p->S;
    int r = (int)(rem % p->R); rem /= p->R;
    int k = (int)rem;
    double sum = 0.0, asum = 0.0;
    for (int n = 0; n < p->N; ++n) {
        for (int pp = 0; pp < t->P; ++pp) {
            int h = pp * p->stride_h - p->pad_h + r * p->dil_h;
            if (h < 0 || h >= p->H) continue;
            for (int q = 0; q < t->Q; ++q) {
                int w = q * p->stride_w - p->pad_w + s * p->dil_w;
                if (w < 0 || w >= p->W) continue;
                double g = t->dY[(((int64_t)n * t->P + pp) * t->Q + q) * p->K + k];
                double x = t->X[(((int64_t)n * p->H + h) * p->W + w) * p->C + c];
                sum += g * x;
                asum += fabs(g * x);
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    t->dW[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

/* idx indexes [K][R][S][C]. */
int oracle_wgrad(const oracle_problem *pb, const double *X, const double *dY,
                 const double *Cin, double alpha, double beta, const int64_t *idx,
                 int64_t count, double *dW, double *A, int nthreads)
{
    wgrad_ctx t;
    t.pb = *pb;
    t.P = oracle_out_size(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
    t.Q = oracle_out_size(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
    if (t.P <= 0 || t.Q <= 0) return -1;
    t.X = X; t.dY = dY; t.Cin = Cin;
    t.alpha = alpha; t.beta = beta;
    t.idx = idx; t.dW = dW; t.A = A;
    oracle_parallel(wgrad_elem, &t, count, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Grouped convolution, all three passes.                                    */
/*   G groups split the C input and K output channels into G equal, ordered  */
/*   runs of Cg = C/G and Kg = K/G channels.  Output channel k belongs to    */
/*   group g = floor(k / Kg) and sees only the input channels                */
/*   g*Cg .. g*Cg + Cg - 1; its filter Wt[k][r][s][j] (j < Cg) holds the      */
/*   weight of input channel g*Cg + j.  G = 1 is the dense convolution above; */
/*   G = C = K is the depthwise convolution.                                 */
/* Sources: burn-cubecl "kernel/conv/base.rs", conv_forward_nhwc            */
/* (`options.groups`, grouped problems leave the implicit GEMM for the      */
/* direct kernel); tensorcore "docs/conv2d.md", "What's not done in v0.1"    */
/* (depthwise = groups equal to the input channel count); apache/tvm PR     */
/* #10177 (depthwise wgrad).  The pages do not spell out which channels a    */
/* group holds; the contiguous-run reading above is the one the weight shape */
/* [K][R][S][C/G] of every framework on the pages implies.                   */
/*   fprop  Y[n,p,q,k]  = relu?( alpha * sum_{r,s,j} X[n,h(p,r),w(q,s),g*Cg+j] */
/*                          * Wt[k,r,s,j] + beta * Cin + bias[k] ), g = k/Kg */
/*   dgrad  dX[n,h,w,c] = alpha * sum over k in group g = c/Cg, taps and     */
/*                        (p,q) reading (h,w), of dY[n,p,q,k]*Wt[k,r,s,c-g*Cg] */
/*                        + beta * Cin                                       */
/*   wgrad  dW[k,r,s,j] = alpha * sum_{n,p,q} dY[n,p,q,k] *                   */
/*                        X[n,h(p,r),w(q,s),g*Cg+j] + beta * Cin, g = k/Kg    */
/* with h(p,r) = p*sh - ph + r*dh and w(q,s) = q*sw - pw + s*dw.             */
/* ------------------------------------------------------------------------ */

typedef struct {
    oracle_problem pb;
    int G, Cg, Kg, P, Q;
    const double *A_in, *B_in, *bias, *Cin;   /* fprop: X, Wt; dgrad: dY, Wt; wgrad: X, dY */
    double alpha, beta;
    int relu;
    const int64_t *idx;
    double *out, *A;
} grouped_ctx;

static void grouped_fprop_elem(const void *vctx, int64_t j)
{
    const grouped_ctx *t = (const grouped_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int k = (int)(rem % p->K); rem /= p->K;
    int q = (int)(rem % t->Q); rem /= t->Q;
    int pp = (int)(rem % t->P); rem /= t->P;
    int n = (int)rem;
    int g = k / t->Kg;
    double sum = 0.0, asum = 0.0;
    for (int r = 0; r < p->R; ++r) {
        int h = pp * p->stride_h - p->pad_h + r * p->dil_h;
        if (h < 0 || h >= p->H) continue;
        for (int s = 0; s < p->S; ++s) {
            int w = q * p->stride_w - p->pad_w + s * p->dil_w;
            if (w < 0 || w >= p->W) continue;
            for (int jj = 0; jj < t->Cg; ++jj) {
                double x = t->A_in[(((int64_t)n * p->H + h) * p->W + w) * p->C + g * t->Cg + jj];
                double f = t->B_in[(((int64_t)k * p->R + r) * p->S + s) * t->Cg + jj];
                sum += x * f;
                asum += fabs(x * f);
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    if (t->bias) v += t->bias[k];
    if (t->relu && v < 0.0) v = 0.0;
    t->out[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

static void grouped_dgrad_elem(const void *vctx, int64_t j)
{
    const grouped_ctx *t = (const grouped_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int c = (int)(rem % p->C); rem /= p->C;
    int w = (int)(rem % p->W); rem /= p->W;
    int h = (int)(rem % p->H); rem /= p->H;
    int n = (int)rem;
    int g = c / t->Cg;
    int jj = c - g * t->Cg;
    double sum = 0.0, asum = 0.0;
    for (int r = 0; r < p->R; ++r) {
        int th = h + p->pad_h - r * p->dil_h;
        if (th < 0 || th % p->stride_h != 0) continue;
        int pp = th / p->stride_h;
        if (pp >= t->P) continue;
        for (int s = 0; s < p->S; ++s) {
            int tw = w + p->pad_w - s * p->dil_w;
            if (tw < 0 || tw % p->stride_w != 0) continue;
            int q = tw / p->stride_w;
            if (q >= t->Q) continue;
            for (int k = g * t->Kg; k < (g + 1) * t->Kg; ++k) {
                double gy = t->A_in[(((int64_t)n * t->P + pp) * t->Q + q) * p->K + k];
                double f = t->B_in[(((int64_t)k * p->R + r) * p->S + s) * t->Cg + jj];
                sum += gy * f;
                asum += fabs(gy * f);
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    t->out[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

static void grouped_wgrad_elem(const void *vctx, int64_t j)
{
    const grouped_ctx *t = (const grouped_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int jj = (int)(rem % t->Cg); rem /= t->Cg;
    int s = (int)(rem % p->S); rem /= p->S;
    int r = (int)(rem % p->R); rem /= p->R;
    int k = (int)rem;
    int c = (k / t->Kg) * t->Cg + jj;
    double sum = 0.0, asum = 0.0;
    for (int n = 0; n < p->N; ++n) {
        for (int pp = 0; pp < t->P; ++pp) {
            int h = pp * p->stride_h - p->pad_h + r * p->dil_h;
            if (h < 0 || h >= p->H) continue;
            for (int q = 0; q < t->Q; ++q) {
                int w = q * p->stride_w - p->pad_w + s * p->dil_w;
                if (w < 0 || w >= p->W) continue;
                double x = t->A_in[(((int64_t)n * p->H + h) * p->W + w) * p->C + c];
                double gy = t->B_in[(((int64_t)n * t->P + pp) * t->Q + q) * p->K + k];
                sum += gy * x;
                asum += fabs(gy * x);
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    t->out[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

/* which: 0 fprop (A_in = X, B_in = Wt, idx into [N][P][Q][K]),
 *        1 dgrad (A_in = dY, B_in = Wt, idx into [N][H][W][C]),
 *        2 wgrad (A_in = X, B_in = dY, idx into [K][R][S][C/G]).
 * bias and relu apply to fprop only.  Returns 0; -1 for an empty output
 * size; -2 when G < 1 or G does not divide both C and K. */
int oracle_grouped(int which, const oracle_problem *pb, int groups, const double *A_in,
                   const double *B_in, const double *bias, const double *Cin, double alpha,
                   double beta, int relu, const int64_t *idx, int64_t count, double *out,
                   double *A, int nthreads)
{
    grouped_ctx t;
    if (groups < 1 || pb->C % groups != 0 || pb->K % groups != 0) return -2;
    t.pb = *pb;
    t.G = groups;
    t.Cg = pb->C / groups;
    t.Kg = pb->K / groups;
    t.P = oracle_out_size(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
    t.Q = oracle_out_size(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
    if (t.P <= 0 || t.Q <= 0) return -1;
    t.A_in = A_in; t.B_in = B_in; t.bias = bias; t.Cin = Cin;
    t.alpha = alpha; t.beta = beta; t.relu = relu;
    t.idx = idx; t.out = out; t.A = A;
    oracle_elem_fn fn = which == 0 ? grouped_fprop_elem
                      : which == 1 ? grouped_dgrad_elem : grouped_wgrad_elem;
    oracle_parallel(fn, &t, count, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 3D fprop (volumes: one more spatial dimension, depth).                    */
/*   Y[n,o,p,q,k] = relu?( alpha * sum_{t,r,s,c} X[n, o*sd - pd + t*dd,      */
/*                          p*sh - ph + r*dh, q*sw - pw + s*dw, c]           */
/*                          * W[k,t,r,s,c] + beta * Cin[n,o,p,q,k] + bias[k] ) */
/* Out-of-range input positions contribute nothing.  Layouts NDHWC (X),      */
/* KTRSC (W), N Do P Q K (Y).  Sources: burn-cubecl "kernel/conv/base.rs"    */
/* (ConvOptions<N>, the same stride/padding/dilation per spatial dimension); */
/* PyTorch quantized cuDNN Conv.cpp (kSpatialDim = 2 or 3).  The output      */
/* extent per dimension is oracle_out_size.                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    int N, D, H, W, C, K, T, R, S;
    int pad_d, pad_h, pad_w, stride_d, stride_h, stride_w, dil_d, dil_h, dil_w;
} oracle_problem3d;

typedef struct {
    oracle_problem3d pb;
    int Do, P, Q;
    const double *X, *Wt, *bias, *Cin;
    double alpha, beta;
    int relu;
    const int64_t *idx;
    double *Y, *A;
} fprop3d_ctx;

static void fprop3d_elem(const void *vctx, int64_t j)
{
    const fprop3d_ctx *t = (const fprop3d_ctx *)vctx;
    const oracle_problem3d *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int k = (int)(rem % p->K); rem /= p->K;
    int q = (int)(rem % t->Q); rem /= t->Q;
    int pp = (int)(rem % t->P); rem /= t->P;
    int o = (int)(rem % t->Do); rem /= t->Do;
    int n = (int)rem;
    double sum = 0.0, asum = 0.0;
    for (int tt = 0; tt < p->T; ++tt) {
        int d = o * p->stride_d - p->pad_d + tt * p->dil_d;
        if (d < 0 || d >= p->D) continue;
        for (int r = 0; r < p->R; ++r) {
            int h = pp * p->stride_h - p->pad_h + r * p->dil_h;
            if (h < 0 || h >= p->H) continue;
            for (int s = 0; s < p->S; ++s) {
                int w = q * p->stride_w - p->pad_w + s * p->dil_w;
                if (w < 0 || w >= p->W) continue;
                for (int c = 0; c < p->C; ++c) {
                    double x = t->X[((((int64_t)n * p->D + d) * p->H + h) * p->W + w) * p->C + c];
                    double f = t->Wt[((((int64_t)k * p->T + tt) * p->R + r) * p->S + s) * p->C + c];
                    sum += x * f;
                    asum += fabs(x * f);
                }
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    if (t->bias) v += t->bias[k];
    if (t->relu && v < 0.0) v = 0.0;
    t->Y[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

/* idx indexes [N][Do][P][Q][K].  Returns 0, or -1 for an empty output. */
int oracle_fprop3d(const oracle_problem3d *pb, const double *X, const double *Wt,
                   const double *bias, const double *Cin, double alpha, double beta, int relu,
                   const int64_t *idx, int64_t count, double *Y, double *A, int nthreads)
{
    fprop3d_ctx t;
    t.pb = *pb;
    t.Do = oracle_out_size(pb->D, pb->pad_d, pb->dil_d, pb->T, pb->stride_d);
    t.P = oracle_out_size(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
    t.Q = oracle_out_size(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
    if (t.Do <= 0 || t.P <= 0 || t.Q <= 0) return -1;
    t.X = X; t.Wt = Wt; t.bias = bias; t.Cin = Cin;
    t.alpha = alpha; t.beta = beta; t.relu = relu;
    t.idx = idx; t.Y = Y; t.A = A;
    oracle_parallel(fprop3d_elem, &t, count, nthreads);
    return 0;
}

/* 3D dgrad and wgrad: the adjoints of fprop3d in X and in W.               */
/*   dX[n,d,h,w,c] = alpha * sum over (k,t,r,s) and the output position      */
/*                   (o,p,q) that reads (d,h,w) through tap (t,r,s), of      */
/*                   dY[n,o,p,q,k] * W[k,t,r,s,c]  +  beta * Cin             */
/*   dW[k,t,r,s,c] = alpha * sum_{n,o,p,q} dY[n,o,p,q,k] *                    */
/*                   X[n, o*sd - pd + t*dd, p*sh - ph + r*dh, q*sw - pw + s*dw, c] */
/*                   + beta * Cin                                            */

typedef struct {
    oracle_problem3d pb;
    int Do, P, Q;
    const double *A_in, *B_in, *Cin;   /* dgrad: dY, W; wgrad: X, dY */
    double alpha, beta;
    const int64_t *idx;
    double *out, *A;
} back3d_ctx;

static void dgrad3d_elem(const void *vctx, int64_t j)
{
    const back3d_ctx *t = (const back3d_ctx *)vctx;
    const oracle_problem3d *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int c = (int)(rem % p->C); rem /= p->C;
    int w = (int)(rem % p->W); rem /= p->W;
    int h = (int)(rem % p->H); rem /= p->H;
    int d = (int)(rem % p->D); rem /= p->D;
    int n = (int)rem;
    double sum = 0.0, asum = 0.0;
    for (int tt = 0; tt < p->T; ++tt) {
        int td = d + p->pad_d - tt * p->dil_d;
        if (td < 0 || td % p->stride_d != 0) continue;
        int o = td / p->stride_d;
        if (o >= t->Do) continue;
        for (int r = 0; r < p->R; ++r) {
            int th = h + p->pad_h - r * p->dil_h;
            if (th < 0 || th % p->stride_h != 0) continue;
            int pp = th / p->stride_h;
            if (pp >= t->P) continue;
            for (int s = 0; s < p->S; ++s) {
                int tw = w + p->pad_w - s * p->dil_w;
                if (tw < 0 || tw % p->stride_w != 0) continue;
                int q = tw / p->stride_w;
                if (q >= t->Q) continue;
                for (int k = 0; k < p->K; ++k) {
                    double g = t->A_in[((((int64_t)n * t->Do + o) * t->P + pp) * t->Q + q) * p->K + k];
                    double f = t->B_in[((((int64_t)k * p->T + tt) * p->R + r) * p->S + s) * p->C + c];
                    sum += g * f;
                    asum += fabs(g * f);
                }
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    t->out[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

static void wgrad3d_elem(const void *vctx, int64_t j)
{
    const back3d_ctx *t = (const back3d_ctx *)vctx;
    const oracle_problem3d *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int c = (int)(rem % p->C); rem /= p->C;
    int s = (int)(rem % p->S); rem /= p->S;
    int r = (int)(rem % p->R); rem /= p->R;
    int tt = (int)(rem % p->T); rem /= p->T;
    int k = (int)rem;
    double sum = 0.0, asum = 0.0;
    for (int n = 0; n < p->N; ++n) {
        for (int o = 0; o < t->Do; ++o) {
            int d = o * p->stride_d - p->pad_d + tt * p->dil_d;
            if (d < 0 || d >= p->D) continue;
            for (int pp = 0; pp < t->P; ++pp) {
                int h = pp * p->stride_h - p->pad_h + r * p->dil_h;
                if (h < 0 || h >= p->H) continue;
                for (int q = 0; q < t->Q; ++q) {
                    int w = q * p->stride_w - p->pad_w + s * p->dil_w;
                    if (w < 0 || w >= p->W) continue;
                    double x = t->A_in[((((int64_t)n * p->D + d) * p->H + h) * p->W + w) * p->C + c];
                    double g = t->B_in[((((int64_t)n * t->Do + o) * t->P + pp) * t->Q + q) * p->K + k];
                    sum += g * x;
                    asum += fabs(g * x);
                }
            }
        }
    }
    double v = t->alpha * sum;
    if (t->beta != 0.0) v += t->beta * t->Cin[e];
    t->out[j] = v;
    if (t->A) t->A[j] = fabs(t->alpha) * asum;
}

/* which: 1 dgrad (A_in = dY, B_in = W, idx into [N][D][H][W][C]),
 *        2 wgrad (A_in = X, B_in = dY, idx into [K][T][R][S][C]). */
int oracle_backward3d(int which, const oracle_problem3d *pb, const double *A_in,
                      const double *B_in, const double *Cin, double alpha, double beta,
                      const int64_t *idx, int64_t count, double *out, double *A, int nthreads)
{
    back3d_ctx t;
    t.pb = *pb;
    t.Do = oracle_out_size(pb->D, pb->pad_d, pb->dil_d, pb->T, pb->stride_d);
    t.P = oracle_out_size(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
    t.Q = oracle_out_size(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
    if (t.Do <= 0 || t.P <= 0 || t.Q <= 0) return -1;
    t.A_in = A_in; t.B_in = B_in; t.Cin = Cin;
    t.alpha = alpha; t.beta = beta;
    t.idx = idx; t.out = out; t.A = A;
    oracle_parallel(which == 1 ? dgrad3d_elem : wgrad3d_elem, &t, count, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* int8 fprop with requantisation                                            */
/*   acc = sum_{r,s,c} X*W            (exact, int64)                         */
/*   t   = acc + bias[k]              (bias in accumulator units)            */
/*   t   = max(t, 0) if relu                                                  */
/*   y   = clamp(round_half_even(t * M), -128, 127),                         */
/*   M   = (float)((act_scale * w_scale) / out_scale)                        */
/* ------------------------------------------------------------------------ */

/* The fp32 requantisation multiplier, from a double quotient as the page
 * computes it from q_scale() doubles. */
float oracle_requant_multiplier(double act_scale, double w_scale, double out_scale)
{
    double m = act_scale * w_scale / out_scale;
    return (float)m;
}

/* t * M is exact in double when |t| < 2^29 (24-bit significand of M times a
 * 29-bit integer fits in 53 bits); nearbyint() in the default rounding mode
 * rounds half to even.  Larger |t| saturates either way for any M >= 2^-21,
 * and is otherwise computed with a split product that is also exact. */
int oracle_requant(int64_t t, float M, int relu)
{
    if (relu && t < 0) t = 0;
    double m = (double)M;
    double prod;
    if (t > -(1LL << 29) && t < (1LL << 29)) {
        prod = (double)t * m;
    } else {
        /* exact split: t = hi * 2^20 + lo, both pieces times m exact */
        int64_t hi = t / (1LL << 20), lo = t - hi * (1LL << 20);
        double ph = (double)hi * m * 1048576.0, pl = (double)lo * m;
        prod = ph + pl; /* may round; only reached far beyond the int8 range */
    }
    double y = nearbyint(prod);
    if (y > 127.0) y = 127.0;
    if (y < -128.0) y = -128.0;
    return (int)y;
}

typedef struct {
    oracle_problem pb;
    int P, Q;
    const int8_t *X, *Wt;
    const int32_t *bias;
    float M;
    int relu;
    const int64_t *idx;
    int8_t *Y;
    int64_t *acc;
} int8_ctx;

static void int8_elem(const void *vctx, int64_t j)
{
    const int8_ctx *t = (const int8_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int k = (int)(rem % p->K); rem /= p->K;
    int q = (int)(rem % t->Q); rem /= t->Q;
    int pp = (int)(rem % t->P); rem /= t->P;
    int n = (int)rem;
    int64_t sum = 0;
    for (int r = 0; r < p->R; ++r) {
        int h = pp * p->stride_h - p->pad_h + r * p->dil_h;
        if (h < 0 || h >= p->H) continue;
        for (int s = 0; s < p->S; ++s) {
            int w = q * p->stride_w - p->pad_w + s * p->dil_w;
            if (w < 0 || w >= p->W) continue;
            for (int c = 0; c < p->C; ++c) {
                int64_t x = t->X[(((int64_t)n * p->H + h) * p->W + w) * p->C + c];
                int64_t f = t->Wt[(((int64_t)k * p->R + r) * p->S + s) * p->C + c];
                sum += x * f;
            }
        }
    }
    if (t->acc) t->acc[j] = sum;
    int64_t v = sum + (t->bias ? (int64_t)t->bias[k] : 0);
    t->Y[j] = (int8_t)oracle_requant(v, t->M, t->relu);
}

int oracle_fprop_int8(const oracle_problem *pb, const int8_t *X, const int8_t *Wt,
                      const int32_t *bias, double act_scale, double w_scale,
                      double out_scale, int relu, const int64_t *idx, int64_t count,
                      int8_t *Y, int64_t *acc, int nthreads)
{
    int8_ctx t;
    t.pb = *pb;
    t.P = oracle_out_size(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
    t.Q = oracle_out_size(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
    if (t.P <= 0 || t.Q <= 0) return -1;
    t.X = X; t.Wt = Wt; t.bias = bias;
    t.M = oracle_requant_multiplier(act_scale, w_scale, out_scale);
    t.relu = relu;
    t.idx = idx; t.Y = Y; t.acc = acc;
    oracle_parallel(int8_elem, &t, count, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* int8 data and weight gradients (int32 results)                            */
/*   dX[n,h,w,c] = sum over (k, r, s) and the output position (p, q) that    */
/*                 reads (h, w) through tap (r, s) of dY[n,p,q,k]*W[k,r,s,c] */
/*   dW[k,r,s,c] = sum_{n,p,q} dY[n,p,q,k] * X[n, p*sh - ph + r*dh,          */
/*                 q*sw - pw + s*dw, c]                                      */
/* int8 operands, the sums taken exactly in int64 and delivered as int32:    */
/* the value modulo 2^32 in two's complement, which is what an int32         */
/* accumulator holds.  Sources: PyTorch quantized cuDNN Conv.cpp (the int8    */
/* convolution computes in INT32; kSpatialDim makes the op generic), and the  */
/* adjoints of fprop written out above.  The pages give no requantisation    */
/* for the backward passes, so none is applied.                              */
/* ------------------------------------------------------------------------ */

typedef struct {
    oracle_problem pb;
    int P, Q;
    const int8_t *A_in, *B_in;
    const int64_t *idx;
    int32_t *out;
    int64_t *acc;
} int8_back_ctx;

static int32_t oracle_wrap_int32(int64_t v)
{
    uint32_t u = (uint32_t)((uint64_t)v & 0xFFFFFFFFu);
    return u >= 0x80000000u ? (int32_t)(int64_t)(u - 0x100000000LL) : (int32_t)u;
}

static void dgrad_int8_elem(const void *vctx, int64_t j)
{
    const int8_back_ctx *t = (const int8_back_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int c = (int)(rem % p->C); rem /= p->C;
    int w = (int)(rem % p->W); rem /= p->W;
    int h = (int)(rem % p->H); rem /= p->H;
    int n = (int)rem;
    int64_t sum = 0;
    for (int r = 0; r < p->R; ++r) {
        int th = h + p->pad_h - r * p->dil_h;
        if (th < 0 || th % p->stride_h != 0) continue;
        int pp = th / p->stride_h;
        if (pp >= t->P) continue;
        for (int s = 0; s < p->S; ++s) {
            int tw = w + p->pad_w - s * p->dil_w;
            if (tw < 0 || tw % p->stride_w != 0) continue;
            int q = tw / p->stride_w;
            if (q >= t->Q) continue;
            for (int k = 0; k < p->K; ++k) {
                int64_t g = t->A_in[(((int64_t)n * t->P + pp) * t->Q + q) * p->K + k];
                int64_t f = t->B_in[(((int64_t)k * p->R + r) * p->S + s) * p->C + c];
                sum += g * f;
            }
        }
    }
    if (t->acc) t->acc[j] = sum;
    t->out[j] = oracle_wrap_int32(sum);
}

static void wgrad_int8_elem(const void *vctx, int64_t j)
{
    const int8_back_ctx *t = (const int8_back_ctx *)vctx;
    const oracle_problem *p = &t->pb;
    int64_t e = t->idx ? t->idx[j] : j;
    int64_t rem = e;
    int c = (int)(rem % p->C); rem /= p->C;
    int s = (int)(rem % p->S); rem /= p->S;
    int r = (int)(rem % p->R); rem /= p->R;
    int k = (int)rem;
    int64_t sum = 0;
    for (int n = 0; n < p->N; ++n) {
        for (int pp = 0; pp < t->P; ++pp) {
            int h = pp * p->stride_h - p->pad_h + r * p->dil_h;
            if (h < 0 || h >= p->H) continue;
            for (int q = 0; q < t->Q; ++q) {
                int w = q * p->stride_w - p->pad_w + s * p->dil_w;
                if (w < 0 || w >= p->W) continue;
                int64_t x = t->A_in[(((int64_t)n * p->H + h) * p->W + w) * p->C + c];
                int64_t g = t->B_in[(((int64_t)n * t->P + pp) * t->Q + q) * p->K + k];
                sum += g * x;
            }
        }
    }
    if (t->acc) t->acc[j] = sum;
    t->out[j] = oracle_wrap_int32(sum);
}

/* which: 1 dgrad (A_in = dY, B_in = W, idx into [N][H][W][C]),
 *        2 wgrad (A_in = X, B_in = dY, idx into [K][R][S][C]).
 * out receives the int32 results; acc (may be NULL) the exact int64 sums. */
int oracle_backward_int8(int which, const oracle_problem *pb, const int8_t *A_in,
                         const int8_t *B_in, const int64_t *idx, int64_t count, int32_t *out,
                         int64_t *acc, int nthreads)
{
    int8_back_ctx t;
    t.pb = *pb;
    t.P = oracle_out_size(pb->H, pb->pad_h, pb->dil_h, pb->R, pb->stride_h);
    t.Q = oracle_out_size(pb->W, pb->pad_w, pb->dil_w, pb->S, pb->stride_w);
    if (t.P <= 0 || t.Q <= 0) return -1;
    if (which != 1 && which != 2) return -2;
    t.A_in = A_in; t.B_in = B_in;
    t.idx = idx; t.out = out; t.acc = acc;
    oracle_parallel(which == 1 ? dgrad_int8_elem : wgrad_int8_elem, &t, count, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Output rounding: double -> IEEE binary16 / bfloat16 bit patterns,         */
/* round to nearest, ties to even, overflow to infinity.                      */
/* Written from the format definitions: binary16 has 10 fraction bits,       */
/* exponent bias 15, minimum normal 2^-14; bfloat16 has 7 fraction bits,     */
/* exponent bias 127, minimum normal 2^-126.                                 */
/* ------------------------------------------------------------------------ */

static uint16_t oracle_round_to_format(double v, int frac_bits, int exp_bias, int exp_bits)
{
    uint16_t sign = signbit(v) ? (uint16_t)(1u << (frac_bits + exp_bits)) : 0;
    uint16_t exp_all_ones = (uint16_t)(((1u << exp_bits) - 1u) << frac_bits);
    if (isnan(v)) return (uint16_t)(exp_all_ones | (1u << (frac_bits - 1)));
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | exp_all_ones);
    if (a == 0.0) return sign;
    int emin = 1 - exp_bias;                   /* exponent of the min normal */
    int e;
    (void)frexp(a, &e);                        /* a = m * 2^e, m in [0.5, 1) */
    int unbiased = e - 1;                      /* a in [2^unbiased, 2^(unbiased+1)) */
    if (unbiased < emin) unbiased = emin;      /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, unbiased - frac_bits);
    double units = nearbyint(a / quantum);     /* exact scaling, RNE */
    double r = units * quantum;                /* the rounded magnitude */
    int emax = exp_bias;                       /* exponent of the max finite */
    double max_finite = ldexp(2.0 - ldexp(1.0, -frac_bits), emax);
    if (r > max_finite) return (uint16_t)(sign | exp_all_ones);
    if (r < ldexp(1.0, emin)) {                /* subnormal: exponent field 0 */
        uint32_t mant = (uint32_t)(r / ldexp(1.0, emin - frac_bits));
        return (uint16_t)(sign | mant);
    }
    int er;
    double mr = frexp(r, &er);                 /* r = mr * 2^er */
    int ub = er - 1;
    uint32_t field = (uint32_t)(ub + exp_bias);
    uint32_t mant = (uint32_t)((mr * 2.0 - 1.0) * ldexp(1.0, frac_bits));
    return (uint16_t)(sign | (field << frac_bits) | mant);
}

uint16_t oracle_f64_to_f16_bits(double v) { return oracle_round_to_format(v, 10, 15, 5); }
uint16_t oracle_f64_to_bf16_bits(double v) { return oracle_round_to_format(v, 7, 127, 8); }

void oracle_round_array(const double *v, int64_t count, int is_bf16, uint16_t *out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = is_bf16 ? oracle_f64_to_bf16_bits(v[i]) : oracle_f64_to_f16_bits(v[i]);
}

/* ------------------------------------------------------------------------ */
/* Permutes (byte copies, any element size)                                  */
/*   nchw_to_nhwc: dst[n][h][w][c] = src[n][c][h][w]                         */
/*   nhwc_to_nchw: dst[n][c][h][w] = src[n][h][w][c]                         */
/* ------------------------------------------------------------------------ */

void oracle_nchw_to_nhwc(const void *src, void *dst, int N, int C, int H, int W, int eb)
{
    const unsigned char *s = (const unsigned char *)src;
    unsigned char *d = (unsigned char *)dst;
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < C; ++c)
            for (int h = 0; h < H; ++h)
                for (int w = 0; w < W; ++w) {
                    int64_t si = (((int64_t)n * C + c) * H + h) * W + w;
                    int64_t di = (((int64_t)n * H + h) * W + w) * C + c;
                    memcpy(d + di * eb, s + si * eb, (size_t)eb);
                }
}

void oracle_nhwc_to_nchw(const void *src, void *dst, int N, int C, int H, int W, int eb)
{
    const unsigned char *s = (const unsigned char *)src;
    unsigned char *d = (unsigned char *)dst;
    for (int n = 0; n < N; ++n)
        for (int h = 0; h < H; ++h)
            for (int w = 0; w < W; ++w)
                for (int c = 0; c < C; ++c) {
                    int64_t si = (((int64_t)n * H + h) * W + w) * C + c;
                    int64_t di = (((int64_t)n * C + c) * H + h) * W + w;
                    memcpy(d + di * eb, s + si * eb, (size_t)eb);
                }
}
