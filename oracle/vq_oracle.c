/*
 * vq_oracle.c -- plain, slow, obviously correct CPU oracle for the
 * product-vector-quantisation encode step ("quantize_vq").
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library and its Python binding) never calls it, and the two
 * share no code, headers, tables or helpers.
 *
 * What it computes (source: "I Wrote a Metal Kernel to Stop My Mac From
 * OOMing", sections "What Even Is a KV Cache" steps 1-3, "What quantize_vq
 * Was Doing Wrong" and "The Kernel: 18 Lines of MSL"):
 *
 *   for every sub-vector x[n] (length sub_dim) and its codebook cb
 *   [n_centroids][sub_dim]:
 *     best = +inf (fp32), idx = 0
 *     for c = 0 .. n_centroids-1 (ascending):
 *       dist = 0 (fp32)
 *       for i = 0 .. sub_dim-1 (ascending):
 *         d    = float(x[n][i]) - float(cb[c][i])     fp32, round to nearest
 *         dist = dist + d * d                           separate fp32 multiply
 *                                                      and add, never fused
 *       if dist < best: best = dist; idx = c           strict "<"
 *     out[n] = idx   (uint32)
 *
 * Readings where the page is silent (each is also listed with the design
 * notes): the multiply and add are not contracted into an FMA (this file
 * must be compiled with -ffp-contract=off and without fast-math); fp16 and
 * bf16 inputs are widened to fp32 before the subtraction (the shader's
 * float(...) casts); a NaN distance never wins and a row whose distances
 * are all NaN or +inf encodes to 0 (consequence of the (+inf, 0) start and
 * the strict compare); denormals are kept (IEEE, no flush to zero).
 *
 * Grouped layout (one codebook per (layer, head) group): x is
 * [n_groups][n_per_group][sub_dim], codebooks [n_groups][n_centroids]
 * [sub_dim], out [n_groups][n_per_group]; row n of the flattened x uses
 * codebook n / n_per_group.  The ungrouped call is n_groups = 1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { VQO_F16 = 0, VQO_BF16 = 1, VQO_F32 = 2 };

enum {
    VQO_OK = 0,
    VQO_ERR_INVALID_ARG = 1,
    VQO_ERR_THREAD = 2
};

/* IEEE 754 binary16 -> binary32, from the format's definition:
 * value = (-1)^s * 2^(e-15) * (1 + m/1024) for 0 < e < 31,
 *         (-1)^s * 2^-14 * (m/1024)          for e == 0,
 *         inf / NaN                          for e == 31.        */
float vqo_f16_to_f32(uint16_t h)
{
    uint32_t s = (h >> 15) & 1u;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t m = h & 0x3ffu;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(m | 0x400u), (int)e - 25);
    return s ? -v : v;
}

/* bfloat16 is the upper half of a binary32. */
float vqo_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float load_elem(const void *base, int dtype, int64_t k)
{
    switch (dtype) {
    case VQO_F16:
        return vqo_f16_to_f32(((const uint16_t *)base)[k]);
    case VQO_BF16:
        return vqo_bf16_to_f32(((const uint16_t *)base)[k]);
    default:
        return ((const float *)base)[k];
    }
}

/* The fp32 formula above for a row x (elements of x_dtype) and a centroid
 * c (elements of c_dtype). */
static float distance_of(const void *x, int x_dtype, const void *c, int c_dtype, int32_t sub_dim)
{
    float dist = 0.0f;
    for (int32_t i = 0; i < sub_dim; ++i) {
        float d = load_elem(x, x_dtype, i) - load_elem(c, c_dtype, i);
        float sq = d * d;
        dist = dist + sq;
    }
    return dist;
}

/* Squared distance of one sub-vector to one centroid, the fp32 formula
 * above.  Exported so the tests can pin the arithmetic on its own. */
float vqo_distance(const void *x, const void *c, int32_t sub_dim, int32_t dtype)
{
    return distance_of(x, dtype, c, dtype, sub_dim);
}

static size_t elem_size(int dtype)
{
    return dtype == VQO_F32 ? 4u : 2u;
}

/* Encode flattened rows [row_begin, row_end).  With smooth != NULL each
 * element is first divided by its channel's smooth factor (fp32, round to
 * nearest): row m of group g holds channels (m % (head_dim / sub_dim)) *
 * sub_dim + i of a key vector, factors smooth[g][head_dim]. */
static void encode_rows(const void *x, const void *codebooks, int64_t n_per_group,
                        int32_t n_centroids, int32_t sub_dim, int32_t dtype,
                        const float *smooth, int32_t head_dim,
                        uint32_t *out, int64_t row_begin, int64_t row_end)
{
    const size_t es = elem_size(dtype);
    const char *xb = (const char *)x;
    const char *cbb = (const char *)codebooks;
    float *xs = smooth ? (float *)malloc((size_t)sub_dim * sizeof(float)) : NULL;
    for (int64_t n = row_begin; n < row_end; ++n) {
        const int64_t g = n / n_per_group;
        const char *xn = xb + (size_t)n * (size_t)sub_dim * es;
        const char *cb = cbb + (size_t)g * (size_t)n_centroids * (size_t)sub_dim * es;
        const void *row = xn;
        int row_dtype = dtype;
        if (xs) {
            const int64_t block = (n - g * n_per_group) % (head_dim / sub_dim);
            const float *f = smooth + (size_t)g * (size_t)head_dim + (size_t)block * (size_t)sub_dim;
            for (int32_t i = 0; i < sub_dim; ++i)
                xs[i] = load_elem(xn, dtype, i) / f[i];
            row = xs;
            row_dtype = VQO_F32;
        }
        float best = INFINITY;
        uint32_t idx = 0;
        for (int32_t c = 0; c < n_centroids; ++c) {
            float dist = distance_of(row, row_dtype, cb + (size_t)c * (size_t)sub_dim * es, dtype,
                                     sub_dim);
            if (dist < best) {
                best = dist;
                idx = (uint32_t)c;
            }
        }
        out[n] = idx;
    }
    free(xs);
}

struct job {
    const void *x;
    const void *codebooks;
    int64_t n_per_group;
    int32_t n_centroids, sub_dim, dtype;
    const float *smooth;
    int32_t head_dim;
    uint32_t *out;
    int64_t begin, end;
};

static void *job_main(void *arg)
{
    struct job *j = (struct job *)arg;
    encode_rows(j->x, j->codebooks, j->n_per_group, j->n_centroids, j->sub_dim, j->dtype,
                j->smooth, j->head_dim, j->out, j->begin, j->end);
    return NULL;
}

/* Encode all n_groups * n_per_group rows with n_threads host threads
 * (rows split into equal contiguous ranges; the result does not depend on
 * the thread count).  Returns VQO_OK or an error code. */
static int32_t encode_all(const void *x, const float *smooth, const void *codebooks,
                          int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                          int32_t sub_dim, int32_t head_dim, int32_t dtype, uint32_t *out,
                          int32_t n_threads)
{
    if (n_groups < 0 || n_per_group < 0 || n_centroids < 1 || sub_dim < 1)
        return VQO_ERR_INVALID_ARG;
    if (dtype != VQO_F16 && dtype != VQO_BF16 && dtype != VQO_F32)
        return VQO_ERR_INVALID_ARG;
    const int64_t rows = n_groups * n_per_group;
    if (rows == 0)
        return VQO_OK;
    if (!x || !codebooks || !out)
        return VQO_ERR_INVALID_ARG;
    if (n_threads < 1)
        n_threads = 1;
    if ((int64_t)n_threads > rows)
        n_threads = (int32_t)rows;
    if (n_threads == 1) {
        encode_rows(x, codebooks, n_per_group, n_centroids, sub_dim, dtype, smooth, head_dim, out,
                    0, rows);
        return VQO_OK;
    }
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof *tid);
    struct job *jobs = (struct job *)calloc((size_t)n_threads, sizeof *jobs);
    if (!tid || !jobs) {
        free(tid);
        free(jobs);
        return VQO_ERR_THREAD;
    }
    int32_t started = 0;
    int32_t rc = VQO_OK;
    for (int32_t t = 0; t < n_threads; ++t) {
        jobs[t] = (struct job){x, codebooks, n_per_group, n_centroids, sub_dim, dtype, smooth,
                               head_dim, out, rows * t / n_threads, rows * (t + 1) / n_threads};
        if (pthread_create(&tid[t], NULL, job_main, &jobs[t]) != 0) {
            rc = VQO_ERR_THREAD;
            break;
        }
        ++started;
    }
    for (int32_t t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    if (rc != VQO_OK) /* finish the rows of threads that never started */
        for (int32_t t = started; t < n_threads; ++t)
            job_main(&jobs[t]);
    free(tid);
    free(jobs);
    return VQO_OK;
}

int32_t vqo_encode_grouped(const void *x, const void *codebooks, int64_t n_groups,
                           int64_t n_per_group, int32_t n_centroids, int32_t sub_dim,
                           int32_t dtype, uint32_t *out, int32_t n_threads)
{
    return encode_all(x, NULL, codebooks, n_groups, n_per_group, n_centroids, sub_dim, sub_dim,
                      dtype, out, n_threads);
}

/* Encode with per-channel smoothing (fused neighbour of the encode: "VecInfer
 * -- 16x with Metal acceleration" on the same site names per-channel smooth
 * scaling for outlier channels; read here as key / factor per channel).
 * smooth: [n_groups][head_dim] fp32; head_dim a multiple of sub_dim and
 * n_per_group a multiple of head_dim / sub_dim (whole key vectors). */
int32_t vqo_encode_grouped_smooth(const void *x, const float *smooth, const void *codebooks,
                                  int64_t n_groups, int64_t n_per_group, int32_t n_centroids,
                                  int32_t sub_dim, int32_t head_dim, int32_t dtype, uint32_t *out,
                                  int32_t n_threads)
{
    if (sub_dim < 1 || head_dim < sub_dim || head_dim % sub_dim != 0 || n_per_group < 0 ||
        n_per_group % (head_dim / sub_dim) != 0)
        return VQO_ERR_INVALID_ARG;
    if (n_groups > 0 && n_per_group > 0 && !smooth)
        return VQO_ERR_INVALID_ARG;
    return encode_all(x, smooth, codebooks, n_groups, n_per_group, n_centroids, sub_dim, head_dim,
                      dtype, out, n_threads);
}

int32_t vqo_encode(const void *x, const void *codebook, int64_t n, int32_t n_centroids,
                   int32_t sub_dim, int32_t dtype, uint32_t *out, int32_t n_threads)
{
    if (n < 0)
        return VQO_ERR_INVALID_ARG;
    return vqo_encode_grouped(x, codebook, 1, n, n_centroids, sub_dim, dtype, out, n_threads);
}

/* ------------------------------------------------------------------------
 * Sibling encoders on the same argmin (the page of five hand-tuned Metal
 * compute kernels for TurboQuant, sections "Kernel 2: Scalar Quantize /
 * Dequantize" and "Kernel 3: Fused Hadamard + Quantize").
 * ---------------------------------------------------------------------- */

/* Nearest scalar centroid of one fp32 value: d = val - c[j], dist = d * d
 * (fp32, round to nearest, separately rounded), strict "<" over ascending j
 * from (+inf, 0). */
static uint32_t scalar_nearest(float val, const float *centroids, int32_t n_centroids)
{
    float best_dist = INFINITY;
    uint32_t best = 0;
    for (int32_t j = 0; j < n_centroids; ++j) {
        float d = val - centroids[j];
        float dist = d * d;
        if (dist < best_dist) {
            best_dist = dist;
            best = (uint32_t)j;
        }
    }
    return best;
}

/* Scalar (sub_dim = 1) quantize of n elements against one fp32 codebook
 * ("Kernel 2"): out[e] = index of the nearest centroid of float(x[e]). */
int32_t vqo_scalar_quantize(const void *x, int32_t dtype, int64_t n, const float *centroids,
                            int32_t n_centroids, uint32_t *out)
{
    if (n < 0 || n_centroids < 1 || (dtype != VQO_F16 && dtype != VQO_BF16 && dtype != VQO_F32))
        return VQO_ERR_INVALID_ARG;
    for (int64_t e = 0; e < n; ++e)
        out[e] = scalar_nearest(load_elem(x, dtype, e), centroids, n_centroids);
    return VQO_OK;
}

/* Randomised Hadamard rotation of rows of length dim (a power of two)
 * ("Kernel 3", steps 1-3): v = float(x) * diag (fp32); for stride = 1, 2,
 * ..., dim/2 every pair (e, e + stride) with e % (2 stride) < stride becomes
 * (v[e] + v[e + stride], v[e] - v[e + stride]) from the previous pass's
 * values (fp32); finally y = v * scale with scale the fp32 value of
 * 1/sqrt(dim) (correctly rounded; the page's rsqrt(float(D))). */
static void hadamard_row(const void *x, int32_t dtype, int64_t row, const float *diag,
                         int32_t dim, float scale, float *v)
{
    for (int32_t e = 0; e < dim; ++e)
        v[e] = load_elem(x, dtype, row * dim + e) * diag[e];
    for (int32_t stride = 1; stride < dim; stride <<= 1) {
        for (int32_t e = 0; e < dim; ++e) {
            if (e % (2 * stride) < stride) {
                const float a = v[e], b = v[e + stride];
                v[e] = a + b;
                v[e + stride] = a - b;
            }
        }
    }
    for (int32_t e = 0; e < dim; ++e)
        v[e] = v[e] * scale;
}

static int dim_ok(int32_t dim)
{
    return dim >= 1 && dim <= 65536 && (dim & (dim - 1)) == 0;
}

/* The rotated rows y [n_rows][dim] (fp32). */
int32_t vqo_hadamard_rotate(const void *x, int32_t dtype, const float *diag, int64_t n_rows,
                            int32_t dim, float scale, float *y)
{
    if (n_rows < 0 || !dim_ok(dim) || (dtype != VQO_F16 && dtype != VQO_BF16 && dtype != VQO_F32))
        return VQO_ERR_INVALID_ARG;
    for (int64_t r = 0; r < n_rows; ++r)
        hadamard_row(x, dtype, r, diag, dim, scale, y + (size_t)r * (size_t)dim);
    return VQO_OK;
}

/* Fused rotation and scalar quantize ("Kernel 3", step 4): out[r][e] = index
 * of the nearest centroid of y[r][e]. */
int32_t vqo_hadamard_quantize(const void *x, int32_t dtype, const float *diag, int64_t n_rows,
                              int32_t dim, float scale, const float *centroids,
                              int32_t n_centroids, uint32_t *out)
{
    if (n_rows < 0 || !dim_ok(dim) || n_centroids < 1 ||
        (dtype != VQO_F16 && dtype != VQO_BF16 && dtype != VQO_F32))
        return VQO_ERR_INVALID_ARG;
    float *v = (float *)malloc((size_t)dim * sizeof(float));
    if (!v)
        return VQO_ERR_THREAD;
    for (int64_t r = 0; r < n_rows; ++r) {
        hadamard_row(x, dtype, r, diag, dim, scale, v);
        for (int32_t e = 0; e < dim; ++e)
            out[(size_t)r * (size_t)dim + (size_t)e] = scalar_nearest(v[e], centroids, n_centroids);
    }
    free(v);
    return VQO_OK;
}
