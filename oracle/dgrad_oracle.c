/*
 * dgrad_oracle.c -- CPU oracle for conv2d's gradient with respect to its input.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Everything here is plain double-precision loops written straight from the
 * definitions, with no blocking, fusion or reordering:
 *
 *  - oracle_dgrad_f64: the gradient of conv2d with respect to its input, as
 *    the adjoint of the forward convolution.  Page
 *    "conv2d_grad_input_gemm_coop.wgsl" (meganeura 0.2.0): its header comment
 *    (per batch item, the input gradient is the transposed weight matrix
 *    times the transposed im2col matrix of grad_out, K = Co*kH*kW) and its
 *    strided staging branch (an input pixel receives grad_out[oh] through
 *    tap kh exactly when ih + padding_h - kh is a non-negative multiple of
 *    the stride whose quotient is a valid output row; the same along w).
 *    Layouts from the same page: grad_out NCHW [N,Co,OH,OW], weight
 *    [Co,Ci,kH,kW], grad_input NCHW [N,Ci,H,W], output overwritten.
 *
 *  - oracle_conv2d_fwd_f64: the forward convolution that the gradient is the
 *    adjoint of, out[n,co,oh,ow] = sum_{ci,kh,kw} x[n,ci,oh*s-ph+kh,ow*s-pw+kw]
 *    * w[co,ci,kh,kw], with x zero outside the image.  It loops over outputs
 *    (the dgrad oracle loops over inputs), so the two are written
 *    independently and the adjoint identity between them is a real check.
 *
 *  - oracle_shader_index_dgrad_f64: the index map the page's shader uses,
 *    restated.  For stride 1 it takes the shortcut oh = ih + (kH-1-ph) - kh
 *    with the weight tap not flipped; for stride > 1 it is the divisibility
 *    test above.  It exists only so the tests can show where the stride-1
 *    shortcut agrees with the definition (kH-1 == 2*ph) and where it does not.
 *
 *  - oracle_dgrad_points_f64: the same definition as oracle_dgrad_f64,
 *    evaluated only at a list of (n, ci, ih, iw) points, for sampled checks
 *    at sizes where the whole tensor would take too long.
 *
 * Parity pins (tests/test_oracle_pins.py): hand-worked fixtures in
 * tests/golden/, closed-form counts for all-ones inputs, torch's CPU float64
 * conv2d / conv2d_input, numpy matmul for the 1x1 case, the adjoint identity,
 * finite differences, and planted mutants that each pin must catch.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

typedef struct {
    int N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW;
} oracle_shape;

/* floor((H + 2p - k) / s) + 1, or 0 when the kernel does not fit at all. */
int oracle_out_size(int in, int k, int pad, int s)
{
    int span = in + 2 * pad - k;
    if (s <= 0 || span < 0) return 0;
    return span / s + 1;
}

static int64_t idx4(int a, int b, int c, int d, int B, int C, int D)
{
    return (((int64_t)a * B + b) * C + c) * D + d;
}

/* ---- the definition: gather into one input pixel ------------------------ */

static double dgrad_one(const double *g, const double *w, const oracle_shape *p,
                        int n, int ci, int ih, int iw)
{
    double acc = 0.0;
    for (int co = 0; co < p->Co; ++co) {
        for (int kh = 0; kh < p->kH; ++kh) {
            int th = ih + p->ph - kh;           /* = s * oh for a contributing tap */
            if (th < 0 || th % p->s != 0) continue;
            int oh = th / p->s;
            if (oh >= p->OH) continue;
            for (int kw = 0; kw < p->kW; ++kw) {
                int tw = iw + p->pw - kw;       /* = s * ow for a contributing tap */
                if (tw < 0 || tw % p->s != 0) continue;
                int ow = tw / p->s;
                if (ow >= p->OW) continue;
                acc += g[idx4(n, co, oh, ow, p->Co, p->OH, p->OW)] *
                       w[idx4(co, ci, kh, kw, p->Ci, p->kH, p->kW)];
            }
        }
    }
    return acc;
}

typedef struct {
    const double *g, *w;
    double *gi;
    const oracle_shape *p;
    int64_t first, last; /* range of (n, ci) planes */
} dgrad_job;

static void *dgrad_worker(void *arg)
{
    const dgrad_job *j = (const dgrad_job *)arg;
    const oracle_shape *p = j->p;
    for (int64_t plane = j->first; plane < j->last; ++plane) {
        int n = (int)(plane / p->Ci), ci = (int)(plane % p->Ci);
        for (int ih = 0; ih < p->H; ++ih)
            for (int iw = 0; iw < p->W; ++iw)
                j->gi[idx4(n, ci, ih, iw, p->Ci, p->H, p->W)] =
                    dgrad_one(j->g, j->w, p, n, ci, ih, iw);
    }
    return NULL;
}

static int pick_threads(int requested, int64_t work_items)
{
    int t = requested;
    if (t <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        t = c > 0 ? (int)c : 1;
    }
    if (t > 256) t = 256;
    if ((int64_t)t > work_items) t = (int)(work_items > 0 ? work_items : 1);
    return t;
}

static int valid_shape(const oracle_shape *p)
{
    if (p->N < 0 || p->Ci < 0 || p->Co < 0 || p->H < 0 || p->W < 0) return 0;
    if (p->kH <= 0 || p->kW <= 0 || p->s <= 0 || p->ph < 0 || p->pw < 0) return 0;
    if (p->OH < 0 || p->OW < 0) return 0;
    return 1;
}

/* Returns the number of threads used, or -1 on a bad shape. */
int oracle_dgrad_f64(const double *grad_out, const double *weight, double *grad_in,
                     int N, int Ci, int H, int W, int Co, int kH, int kW,
                     int s, int ph, int pw, int OH, int OW, int nthreads)
{
    oracle_shape p = {N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW};
    if (!valid_shape(&p)) return -1;
    int64_t planes = (int64_t)N * Ci;
    int t = pick_threads(nthreads, planes);
    pthread_t tid[256];
    dgrad_job jobs[256];
    for (int i = 0; i < t; ++i) {
        jobs[i].g = grad_out; jobs[i].w = weight; jobs[i].gi = grad_in; jobs[i].p = &p;
        jobs[i].first = planes * i / t;
        jobs[i].last = planes * (i + 1) / t;
    }
    int started = 0;
    for (int i = 1; i < t; ++i) {
        if (pthread_create(&tid[i], NULL, dgrad_worker, &jobs[i]) != 0) break;
        started = i;
    }
    /* Any job whose thread did not start runs here, serially. */
    dgrad_worker(&jobs[0]);
    for (int i = started + 1; i < t; ++i) dgrad_worker(&jobs[i]);
    for (int i = 1; i <= started; ++i) pthread_join(tid[i], NULL);
    return t;
}

/* points: npts rows of (n, ci, ih, iw); out[i] = grad_in at that point. */
int oracle_dgrad_points_f64(const double *grad_out, const double *weight,
                            const int64_t *points, int64_t npts, double *out,
                            int N, int Ci, int H, int W, int Co, int kH, int kW,
                            int s, int ph, int pw, int OH, int OW)
{
    oracle_shape p = {N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW};
    if (!valid_shape(&p)) return -1;
    for (int64_t i = 0; i < npts; ++i) {
        int n = (int)points[4 * i], ci = (int)points[4 * i + 1];
        int ih = (int)points[4 * i + 2], iw = (int)points[4 * i + 3];
        if (n < 0 || n >= N || ci < 0 || ci >= Ci || ih < 0 || ih >= H || iw < 0 || iw >= W)
            return -2;
        out[i] = dgrad_one(grad_out, weight, &p, n, ci, ih, iw);
    }
    return 0;
}

/* ---- the forward convolution: loop over outputs, gather inputs ----------- */

int oracle_conv2d_fwd_f64(const double *x, const double *weight, double *out,
                          int N, int Ci, int H, int W, int Co, int kH, int kW,
                          int s, int ph, int pw, int OH, int OW)
{
    oracle_shape p = {N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW};
    if (!valid_shape(&p)) return -1;
    for (int n = 0; n < N; ++n)
        for (int co = 0; co < Co; ++co)
            for (int oh = 0; oh < OH; ++oh)
                for (int ow = 0; ow < OW; ++ow) {
                    double acc = 0.0;
                    for (int ci = 0; ci < Ci; ++ci)
                        for (int kh = 0; kh < kH; ++kh) {
                            int y = oh * s - ph + kh;
                            if (y < 0 || y >= H) continue;
                            for (int kw = 0; kw < kW; ++kw) {
                                int xx = ow * s - pw + kw;
                                if (xx < 0 || xx >= W) continue;
                                acc += x[idx4(n, ci, y, xx, Ci, H, W)] *
                                       weight[idx4(co, ci, kh, kw, Ci, kH, kW)];
                            }
                        }
                    out[idx4(n, co, oh, ow, Co, OH, OW)] = acc;
                }
    return 0;
}

/* ---- the page's index map, restated (documents the stride-1 shortcut) ---- */

int oracle_shader_index_dgrad_f64(const double *grad_out, const double *weight,
                                  double *grad_in, int N, int Ci, int H, int W,
                                  int Co, int kH, int kW, int s, int ph, int pw,
                                  int OH, int OW)
{
    oracle_shape p = {N, Ci, H, W, Co, kH, kW, s, ph, pw, OH, OW};
    if (!valid_shape(&p)) return -1;
    int sh_h = kH - 1 - ph, sh_w = kW - 1 - pw; /* the shortcut's shifted padding */
    for (int n = 0; n < N; ++n)
        for (int ci = 0; ci < Ci; ++ci)
            for (int ih = 0; ih < H; ++ih)
                for (int iw = 0; iw < W; ++iw) {
                    double acc = 0.0;
                    for (int co = 0; co < Co; ++co)
                        for (int kh = 0; kh < kH; ++kh)
                            for (int kw = 0; kw < kW; ++kw) {
                                int oh, ow;
                                if (s == 1) {
                                    oh = ih + sh_h - kh;
                                    ow = iw + sh_w - kw;
                                    if (oh < 0 || ow < 0) continue;
                                } else {
                                    int hh = ih + ph - kh, ww = iw + pw - kw;
                                    if (hh < 0 || ww < 0 || hh % s || ww % s) continue;
                                    oh = hh / s;
                                    ow = ww / s;
                                }
                                if (oh >= OH || ow >= OW) continue;
                                acc += grad_out[idx4(n, co, oh, ow, Co, OH, OW)] *
                                       weight[idx4(co, ci, kh, kw, Ci, kH, kW)];
                            }
                    grad_in[idx4(n, ci, ih, iw, Ci, H, W)] = acc;
                }
    return 0;
}
