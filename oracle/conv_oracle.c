/*
 * CPU oracle for the convolution forward pass.  TEST INFRASTRUCTURE ONLY:
 * the tests, the package smoke check and the benchmark's CPU-baseline leg may
 * call it; the library's compute path never does.
 *
 * What it computes is the plain definition of a (grouped) cross-correlation
 * with stride, symmetric zero padding and dilation, as stated on the page
 * "composable_kernel dispatcher/heuristics/LEARNINGS_GROUPED_CONV.md", introduction
 * (NHWGC x GKYXC -> NHWGK forward) and section 2 (3D shapes, dilation_d/h/w), and
 * on the page "[ET-VK] conv1d runs at ~3% of the GPU's matmul throughput ...",
 * "Measurements" (conv1d shapes, output lengths) and "The conv2d path already
 * solves this" (a GELU after each conv):
 *
 *   out[n,od,oh,ow,g,k] = bias[g,k]
 *       + sum_{z,y,x,c} x[n, od*sd - pd + z*dd, oh*sh - ph + y*dh, ow*sw - pw + x*dw, g, c]
 *                     * w[g, k, z, y, x, c]
 *
 * Taps that fall outside the input read zero.  Optionally GELU(v) = v * Phi(v)
 * with the exact normal CDF, Phi(v) = (1 + erf(v / sqrt 2)) / 2.
 *
 * Layouts (channels last): x is N D H W G C, w is G K Z Y X C, out is
 * N Do Ho Wo G K, bias is G*K.  A 1D problem is the case D = H = 1, a 2D problem
 * the case D = 1.  Output size per spatial dimension:
 *   O = floor((I + 2*pad - dil*(F-1) - 1) / stride) + 1.
 *
 * Arithmetic: inputs arrive as float32 (bf16 and fp32 values are both exact
 * float32 values); every product and sum is formed in double.  Besides the
 * output, the oracle returns S = sum |x*w| over the receptive field, the
 * scale of the per-element error bound.
 *
 * Parallelism: independent output pixels are split across pthreads (a conv1d has
 * a single output row per sample, so rows alone would leave one thread); each
 * output is still one plain loop, so the arithmetic does not depend on the thread
 * count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t N, G, C, K;
    int64_t D, H, W;        /* input spatial */
    int64_t Z, Y, X;        /* filter */
    int64_t sd, sh, sw;     /* stride */
    int64_t pd, ph, pw;     /* padding (both sides) */
    int64_t dd, dh, dw;     /* dilation */
    int64_t Do, Ho, Wo;     /* output spatial */
} oracle_geom;

/* Output length of one spatial dimension; <= 0 means the problem is empty. */
int64_t oracle_out_len(int64_t in, int64_t filt, int64_t stride, int64_t pad, int64_t dil)
{
    int64_t span = in + 2 * pad - dil * (filt - 1) - 1;
    if (span < 0) return 0;
    return span / stride + 1;
}

static int fill_geom(oracle_geom* g, const int64_t* p)
{
    /* p: N G C K D H W Z Y X sd sh sw pd ph pw dd dh dw */
    g->N = p[0]; g->G = p[1]; g->C = p[2]; g->K = p[3];
    g->D = p[4]; g->H = p[5]; g->W = p[6];
    g->Z = p[7]; g->Y = p[8]; g->X = p[9];
    g->sd = p[10]; g->sh = p[11]; g->sw = p[12];
    g->pd = p[13]; g->ph = p[14]; g->pw = p[15];
    g->dd = p[16]; g->dh = p[17]; g->dw = p[18];
    g->Do = oracle_out_len(g->D, g->Z, g->sd, g->pd, g->dd);
    g->Ho = oracle_out_len(g->H, g->Y, g->sh, g->ph, g->dh);
    g->Wo = oracle_out_len(g->W, g->X, g->sw, g->pw, g->dw);
    if (g->Do <= 0 || g->Ho <= 0 || g->Wo <= 0) return -1;
    return 0;
}

static double gelu_exact(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

/* One output element: the definition written out. */
static void one_output(const oracle_geom* g, const float* x, const float* w, const float* bias,
                       int gelu, int64_t n, int64_t od, int64_t oh, int64_t ow, int64_t gi,
                       int64_t k, double* out, double* absum)
{
    double acc = 0.0, s = 0.0;
    for (int64_t z = 0; z < g->Z; ++z) {
        int64_t id = od * g->sd - g->pd + z * g->dd;
        if (id < 0 || id >= g->D) continue;
        for (int64_t y = 0; y < g->Y; ++y) {
            int64_t ih = oh * g->sh - g->ph + y * g->dh;
            if (ih < 0 || ih >= g->H) continue;
            for (int64_t xx = 0; xx < g->X; ++xx) {
                int64_t iw = ow * g->sw - g->pw + xx * g->dw;
                if (iw < 0 || iw >= g->W) continue;
                const float* xp = x + ((((n * g->D + id) * g->H + ih) * g->W + iw) * g->G + gi) * g->C;
                const float* wp = w + ((((gi * g->K + k) * g->Z + z) * g->Y + y) * g->X + xx) * g->C;
                for (int64_t c = 0; c < g->C; ++c) {
                    double prod = (double)xp[c] * (double)wp[c];
                    acc += prod;
                    s += fabs(prod);
                }
            }
        }
    }
    if (bias) acc += (double)bias[gi * g->K + k];
    *out = gelu ? gelu_exact(acc) : acc;
    if (absum) *absum = s;
}

typedef struct {
    const oracle_geom* g;
    const float *x, *w, *bias;
    int gelu;
    double *out, *absum;
    int64_t pix_begin, pix_end;   /* output pixels (n, od, oh, ow), flattened */
} job;

static void* run_pixels(void* arg)
{
    job* j = (job*)arg;
    const oracle_geom* g = j->g;
    for (int64_t q = j->pix_begin; q < j->pix_end; ++q) {
        int64_t ow = q % g->Wo, t = q / g->Wo;
        int64_t oh = t % g->Ho;
        t /= g->Ho;
        int64_t od = t % g->Do, n = t / g->Do;
        for (int64_t gi = 0; gi < g->G; ++gi)
            for (int64_t k = 0; k < g->K; ++k) {
                int64_t e = (q * g->G + gi) * g->K + k;
                one_output(g, j->x, j->w, j->bias, j->gelu, n, od, oh, ow, gi, k,
                           &j->out[e], j->absum ? &j->absum[e] : NULL);
            }
    }
    return NULL;
}

/*
 * Full forward.  params: 19 int64 (see fill_geom).  out, absum: N*Do*Ho*Wo*G*K
 * doubles (absum may be NULL).  bias may be NULL.  Returns 0, or -1 for an empty
 * output / bad thread count.
 */
int oracle_conv_fwd(const int64_t* params, const float* x, const float* w, const float* bias,
                    int gelu, double* out, double* absum, int nthreads)
{
    oracle_geom g;
    if (fill_geom(&g, params)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    int64_t pixels = g.N * g.Do * g.Ho * g.Wo;
    if (nthreads > pixels) nthreads = (int)pixels;
    pthread_t th[256];
    job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].g = &g; jobs[i].x = x; jobs[i].w = w; jobs[i].bias = bias; jobs[i].gelu = gelu;
        jobs[i].out = out; jobs[i].absum = absum;
        jobs[i].pix_begin = pixels * i / nthreads;
        jobs[i].pix_end = pixels * (i + 1) / nthreads;
    }
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, run_pixels, &jobs[i]);
    run_pixels(&jobs[0]);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
    return 0;
}

/*
 * Selected outputs only.  idx: npts rows of (n, od, oh, ow, g, k).  Used where the
 * whole output is too large to compute on the CPU.  Returns -1 on a bad index.
 */
int oracle_conv_fwd_points(const int64_t* params, const float* x, const float* w, const float* bias,
                           int gelu, const int64_t* idx, int64_t npts, double* out, double* absum)
{
    oracle_geom g;
    if (fill_geom(&g, params)) return -1;
    for (int64_t p = 0; p < npts; ++p) {
        const int64_t* q = idx + 6 * p;
        if (q[0] < 0 || q[0] >= g.N || q[1] < 0 || q[1] >= g.Do || q[2] < 0 || q[2] >= g.Ho ||
            q[3] < 0 || q[3] >= g.Wo || q[4] < 0 || q[4] >= g.G || q[5] < 0 || q[5] >= g.K)
            return -1;
        one_output(&g, x, w, bias, gelu, q[0], q[1], q[2], q[3], q[4], q[5], &out[p],
                   absum ? &absum[p] : NULL);
    }
    return 0;
}

/* GELU alone, for pinning against closed-form values. */
void oracle_gelu(const double* v, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = gelu_exact(v[i]);
}

/*
 * Backward passes of the same convolution (the "bwd_data" and "bwd_weight" variants that
 * the page "composable_kernel dispatcher/heuristics/LEARNINGS_GROUPED_CONV.md", section 6,
 * names for the same NHWGC / GKYXC / NHWGK layouts).  Given dy, the gradient of a loss with
 * respect to the forward output (N Do Ho Wo G K), these are the gradients with respect to x
 * and w of the linear map x, w -> sum x*w written above (bias and GELU are outside it):
 *
 *   dx[n,i,g,c] = sum over k and taps t of dy[n,o,g,k] * w[g,k,t,c], over the (t, o) with
 *                 o*s - p + t*d = i in every spatial dimension (o in range)
 *   dw[g,k,t,c] = sum over n and output positions o of dy[n,o,g,k] * x[n, o*s - p + t*d, g, c],
 *                 over the o whose input position is in range
 *
 * Each is written out from its own definition: dx solves o = (i + p - t*d) / s for every tap
 * and keeps the exact, in-range quotients; dw walks every output position per tap.  Both
 * return S = sum |products| per element, as the forward does.
 */

/* the output position that tap t maps onto input position i in one dimension, or -1 */
static int64_t source_pos(int64_t i, int64_t t, int64_t s, int64_t p, int64_t d, int64_t O)
{
    int64_t num = i + p - t * d;
    if (num < 0 || num % s != 0) return -1;
    int64_t o = num / s;
    return o < O ? o : -1;
}

static void one_dx(const oracle_geom* g, const float* dy, const float* w, int64_t n, int64_t id,
                   int64_t ih, int64_t iw, int64_t gi, int64_t c, double* out, double* absum)
{
    double acc = 0.0, s = 0.0;
    for (int64_t z = 0; z < g->Z; ++z) {
        int64_t od = source_pos(id, z, g->sd, g->pd, g->dd, g->Do);
        if (od < 0) continue;
        for (int64_t y = 0; y < g->Y; ++y) {
            int64_t oh = source_pos(ih, y, g->sh, g->ph, g->dh, g->Ho);
            if (oh < 0) continue;
            for (int64_t xx = 0; xx < g->X; ++xx) {
                int64_t ow = source_pos(iw, xx, g->sw, g->pw, g->dw, g->Wo);
                if (ow < 0) continue;
                const float* dyp = dy + ((((n * g->Do + od) * g->Ho + oh) * g->Wo + ow) * g->G + gi) * g->K;
                for (int64_t k = 0; k < g->K; ++k) {
                    double prod = (double)dyp[k] *
                                  (double)w[((((gi * g->K + k) * g->Z + z) * g->Y + y) * g->X + xx) * g->C + c];
                    acc += prod;
                    s += fabs(prod);
                }
            }
        }
    }
    *out = acc;
    if (absum) *absum = s;
}

static void one_dw(const oracle_geom* g, const float* x, const float* dy, int64_t gi, int64_t k, int64_t z,
                   int64_t y, int64_t xx, int64_t c, double* out, double* absum)
{
    double acc = 0.0, s = 0.0;
    for (int64_t n = 0; n < g->N; ++n)
        for (int64_t od = 0; od < g->Do; ++od) {
            int64_t id = od * g->sd - g->pd + z * g->dd;
            if (id < 0 || id >= g->D) continue;
            for (int64_t oh = 0; oh < g->Ho; ++oh) {
                int64_t ih = oh * g->sh - g->ph + y * g->dh;
                if (ih < 0 || ih >= g->H) continue;
                for (int64_t ow = 0; ow < g->Wo; ++ow) {
                    int64_t iw = ow * g->sw - g->pw + xx * g->dw;
                    if (iw < 0 || iw >= g->W) continue;
                    double prod = (double)dy[((((n * g->Do + od) * g->Ho + oh) * g->Wo + ow) * g->G + gi) * g->K + k] *
                                  (double)x[((((n * g->D + id) * g->H + ih) * g->W + iw) * g->G + gi) * g->C + c];
                    acc += prod;
                    s += fabs(prod);
                }
            }
        }
    *out = acc;
    if (absum) *absum = s;
}

typedef struct {
    const oracle_geom* g;
    const float *a, *b;     /* dx: dy, w;  dw: x, dy */
    double *out, *absum;
    int64_t begin, end;     /* dx: input pixels (n, id, ih, iw);  dw: (g, k) pairs */
} bwd_job;

static void* run_dx_pixels(void* arg)
{
    bwd_job* j = (bwd_job*)arg;
    const oracle_geom* g = j->g;
    for (int64_t q = j->begin; q < j->end; ++q) {
        int64_t iw = q % g->W, t = q / g->W;
        int64_t ih = t % g->H;
        t /= g->H;
        int64_t id = t % g->D, n = t / g->D;
        for (int64_t gi = 0; gi < g->G; ++gi)
            for (int64_t c = 0; c < g->C; ++c) {
                int64_t e = (q * g->G + gi) * g->C + c;
                one_dx(g, j->a, j->b, n, id, ih, iw, gi, c, &j->out[e], j->absum ? &j->absum[e] : NULL);
            }
    }
    return NULL;
}

static void* run_dw_pairs(void* arg)
{
    bwd_job* j = (bwd_job*)arg;
    const oracle_geom* g = j->g;
    const int64_t per = g->Z * g->Y * g->X * g->C;
    for (int64_t r = j->begin; r < j->end; ++r) {
        int64_t gi = r / g->K, k = r % g->K;
        for (int64_t z = 0; z < g->Z; ++z)
            for (int64_t y = 0; y < g->Y; ++y)
                for (int64_t xx = 0; xx < g->X; ++xx)
                    for (int64_t c = 0; c < g->C; ++c) {
                        int64_t e = r * per + ((z * g->Y + y) * g->X + xx) * g->C + c;
                        one_dw(g, j->a, j->b, gi, k, z, y, xx, c, &j->out[e], j->absum ? &j->absum[e] : NULL);
                    }
    }
    return NULL;
}

static int run_bwd(const int64_t* params, const float* a, const float* b, double* out, double* absum,
                   int nthreads, int weight)
{
    oracle_geom g;
    if (fill_geom(&g, params)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    int64_t rows = weight ? g.G * g.K : g.N * g.D * g.H * g.W;
    if (nthreads > rows) nthreads = (int)rows;
    pthread_t th[256];
    bwd_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].g = &g; jobs[i].a = a; jobs[i].b = b; jobs[i].out = out; jobs[i].absum = absum;
        jobs[i].begin = rows * i / nthreads;
        jobs[i].end = rows * (i + 1) / nthreads;
    }
    void* (*fn)(void*) = weight ? run_dw_pairs : run_dx_pixels;
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, fn, &jobs[i]);
    fn(&jobs[0]);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
    return 0;
}

/* Backward data.  dy: N Do Ho Wo G K; w: G K Z Y X C; dx, absum: N D H W G C doubles. */
int oracle_conv_bwd_data(const int64_t* params, const float* dy, const float* w, double* dx, double* absum,
                         int nthreads)
{
    return run_bwd(params, dy, w, dx, absum, nthreads, 0);
}

/* Backward weight.  x: N D H W G C; dy: N Do Ho Wo G K; dw, absum: G K Z Y X C doubles. */
int oracle_conv_bwd_weight(const int64_t* params, const float* x, const float* dy, double* dw, double* absum,
                           int nthreads)
{
    return run_bwd(params, x, dy, dw, absum, nthreads, 1);
}

/* Selected elements only (rows of n, d, h, w, g, c for dx; g, k, z, y, x, c for dw). */
int oracle_conv_bwd_points(const int64_t* params, const float* a, const float* b, int weight, const int64_t* idx,
                           int64_t npts, double* out, double* absum)
{
    oracle_geom g;
    if (fill_geom(&g, params)) return -1;
    for (int64_t p = 0; p < npts; ++p) {
        const int64_t* q = idx + 6 * p;
        if (weight) {
            if (q[0] < 0 || q[0] >= g.G || q[1] < 0 || q[1] >= g.K || q[2] < 0 || q[2] >= g.Z || q[3] < 0 ||
                q[3] >= g.Y || q[4] < 0 || q[4] >= g.X || q[5] < 0 || q[5] >= g.C)
                return -1;
            one_dw(&g, a, b, q[0], q[1], q[2], q[3], q[4], q[5], &out[p], absum ? &absum[p] : NULL);
        } else {
            if (q[0] < 0 || q[0] >= g.N || q[1] < 0 || q[1] >= g.D || q[2] < 0 || q[2] >= g.H || q[3] < 0 ||
                q[3] >= g.W || q[4] < 0 || q[4] >= g.G || q[5] < 0 || q[5] >= g.C)
                return -1;
            one_dx(&g, a, b, q[0], q[1], q[2], q[3], q[4], q[5], &out[p], absum ? &absum[p] : NULL);
        }
    }
    return 0;
}
