/*
 * oracle.c -- slow, plain, fp64 CPU oracle for the fused conv2d -> BatchNorm
 * -> SiLU layer.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark are the only code allowed to load it.  It
 * shares nothing with the CUDA library (no header, no helper, no table).
 *
 * What it follows ("Fusing an Epilogue", kernels book):
 *   - section "The problem": the layer is a convolution, then batch
 *     normalisation (a per-channel multiply and add), then SiLU, x * sigmoid(x);
 *   - section "The shape of it": after the K loop the accumulator is scaled
 *     and shifted per output channel (acc * bn_scale + bn_bias) and then
 *     multiplied by its own sigmoid.
 * The page prints no convolution formula; this file writes out the textbook
 * definition (a cross-correlation with zero padding, dilation 1, groups 1,
 * output size floor((H + 2*pad - R)/stride) + 1).  Layouts are NHWC for
 * activations and KRSC for weights; values arrive as raw bf16 bit patterns
 * and are decoded exactly to double.  Everything is accumulated in double,
 * in the order the definition is written (r, then s, then c), without
 * blocking or reordering.
 *
 * The BN fold (gamma, beta, running mean/var, eps -> per-channel scale/bias)
 * and the SiLU itself are in the Python half of the oracle (oracle/__init__.py).
 *
 * Threads: output rows (n, ho) -- or, for the sampled entry point, output
 * pixels -- are split between POSIX threads.  Each output value is still
 * computed by one thread with the same serial sum, so the thread count never
 * changes a result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const double *x;  /* [n][h][w][c] decoded */
    const double *w;  /* [k][r][s][c] decoded */
    int64_t n, h, wi, c, k, r, s;
    int64_t sh, sw, ph, pw, ho, wo;
} conv_problem;

/* One output value of the convolution: the plain 3-deep sum over (r, s, c). */
static double conv_point(const conv_problem *p, int64_t n, int64_t oh, int64_t ow, int64_t k)
{
    double acc = 0.0;
    for (int64_t r = 0; r < p->r; ++r) {
        int64_t ih = oh * p->sh - p->ph + r;
        if (ih < 0 || ih >= p->h) continue;          /* zero padding */
        for (int64_t s = 0; s < p->s; ++s) {
            int64_t iw = ow * p->sw - p->pw + s;
            if (iw < 0 || iw >= p->wi) continue;     /* zero padding */
            const double *xp = p->x + ((n * p->h + ih) * p->wi + iw) * p->c;
            const double *wp = p->w + ((k * p->r + r) * p->s + s) * p->c;
            for (int64_t c = 0; c < p->c; ++c) acc += xp[c] * wp[c];
        }
    }
    return acc;
}

typedef struct {
    const conv_problem *p;
    double *out;
    const int64_t *pixels; /* NULL: all output rows */
    int64_t first, last;   /* half-open range of rows (n*ho) or of pixel list entries */
} conv_job;

static void *conv_rows_worker(void *arg)
{
    conv_job *j = (conv_job *)arg;
    const conv_problem *p = j->p;
    for (int64_t row = j->first; row < j->last; ++row) {
        int64_t n = row / p->ho, oh = row % p->ho;
        for (int64_t ow = 0; ow < p->wo; ++ow) {
            double *o = j->out + ((n * p->ho + oh) * p->wo + ow) * p->k;
            for (int64_t k = 0; k < p->k; ++k) o[k] = conv_point(p, n, oh, ow, k);
        }
    }
    return NULL;
}

static void *conv_pixels_worker(void *arg)
{
    conv_job *j = (conv_job *)arg;
    const conv_problem *p = j->p;
    for (int64_t i = j->first; i < j->last; ++i) {
        int64_t m = j->pixels[i];
        int64_t ow = m % p->wo, oh = (m / p->wo) % p->ho, n = m / (p->wo * p->ho);
        double *o = j->out + i * p->k;
        for (int64_t k = 0; k < p->k; ++k) o[k] = conv_point(p, n, oh, ow, k);
    }
    return NULL;
}

/* Split [0, total) into nthreads contiguous chunks and run worker on each. */
static int run_threads(void *(*worker)(void *), const conv_problem *p, double *out,
                       const int64_t *pixels, int64_t total, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > total) nthreads = total > 0 ? (int)total : 1;
    pthread_t tid[256];
    conv_job jobs[256];
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].p = p;
        jobs[t].out = out;
        jobs[t].pixels = pixels;
        jobs[t].first = total * t / nthreads;
        jobs[t].last = total * (t + 1) / nthreads;
        if (nthreads == 1) {
            worker(&jobs[t]);
        } else if (pthread_create(&tid[t], NULL, worker, &jobs[t]) != 0) {
            rc = -1;
            break;
        } else {
            started++;
        }
    }
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    return rc;
}

/* Decode the two operand tensors and fill the problem description. */
static int setup(conv_problem *p, double **xd, double **wd,
                 const uint16_t *x_bits, const uint16_t *w_bits,
                 int64_t n, int64_t h, int64_t wi, int64_t c, int64_t k, int64_t r, int64_t s,
                 int64_t sh, int64_t sw, int64_t ph, int64_t pw)
{
    if (n < 0 || h < 1 || wi < 1 || c < 1 || k < 0 || r < 1 || s < 1 || sh < 1 || sw < 1 ||
        ph < 0 || pw < 0)
        return -1;
    int64_t ho = (h + 2 * ph - r) / sh + 1, wo = (wi + 2 * pw - s) / sw + 1;
    if (h + 2 * ph < r || wi + 2 * pw < s || ho < 1 || wo < 1) return -1;
    int64_t nx = n * h * wi * c, nw = k * r * s * c;
    *xd = (double *)malloc((size_t)(nx > 0 ? nx : 1) * sizeof(double));
    *wd = (double *)malloc((size_t)(nw > 0 ? nw : 1) * sizeof(double));
    if (!*xd || !*wd) {
        free(*xd);
        free(*wd);
        return -2;
    }
    for (int64_t i = 0; i < nx; ++i) (*xd)[i] = bf16_bits_to_double(x_bits[i]);
    for (int64_t i = 0; i < nw; ++i) (*wd)[i] = bf16_bits_to_double(w_bits[i]);
    p->x = *xd;
    p->w = *wd;
    p->n = n; p->h = h; p->wi = wi; p->c = c; p->k = k; p->r = r; p->s = s;
    p->sh = sh; p->sw = sw; p->ph = ph; p->pw = pw; p->ho = ho; p->wo = wo;
    return 0;
}

/*
 * Full convolution: out[n][ho][wo][k] (double, NHWC), from bf16 bit patterns
 * x[n][h][w][c] and w[k][r][s][c].  Returns 0, or -1 for an invalid shape,
 * -2 when memory runs out.
 */
int oracle_conv2d(const uint16_t *x_bits, const uint16_t *w_bits,
                  int64_t n, int64_t h, int64_t wi, int64_t c, int64_t k, int64_t r, int64_t s,
                  int64_t sh, int64_t sw, int64_t ph, int64_t pw, double *out, int nthreads)
{
    conv_problem p;
    double *xd = NULL, *wd = NULL;
    int rc = setup(&p, &xd, &wd, x_bits, w_bits, n, h, wi, c, k, r, s, sh, sw, ph, pw);
    if (rc) return rc;
    rc = run_threads(conv_rows_worker, &p, out, NULL, n * p.ho, nthreads);
    free(xd);
    free(wd);
    return rc;
}

/*
 * The same convolution at a list of output pixels only: pixel m is the flat
 * index n*ho*wo + oh*wo + ow; out[i][k] receives all k channels of pixel
 * pixels[i].  Used to check very large layers at sampled positions.
 */
int oracle_conv2d_at(const uint16_t *x_bits, const uint16_t *w_bits,
                     int64_t n, int64_t h, int64_t wi, int64_t c, int64_t k, int64_t r, int64_t s,
                     int64_t sh, int64_t sw, int64_t ph, int64_t pw,
                     const int64_t *pixels, int64_t count, double *out, int nthreads)
{
    conv_problem p;
    double *xd = NULL, *wd = NULL;
    int rc = setup(&p, &xd, &wd, x_bits, w_bits, n, h, wi, c, k, r, s, sh, sw, ph, pw);
    if (rc) return rc;
    for (int64_t i = 0; i < count; ++i)
        if (pixels[i] < 0 || pixels[i] >= n * p.ho * p.wo) {
            free(xd);
            free(wd);
            return -1;
        }
    rc = run_threads(conv_pixels_worker, &p, out, pixels, count, nthreads);
    free(xd);
    free(wd);
    return rc;
}
