/*
 * CPU oracle for the fused AllReduce + residual-add + RMSNorm epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link
 * or call this file; only the test suite, the smoke check and the bench's
 * CPU-baseline / reference arm use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (per row i of m rows, element j of H):
 *
 *   1. acc = f32(p_0[i,j]); acc = acc + f32(p_k[i,j]) for k = 1 .. n-1,
 *      every add an IEEE fp32 add rounded to nearest even, strictly in the
 *      rank order of the pointer array.
 *      Source: ROCm/aiter #3817 "perf: optimize fused AllReduce + RMSNorm
 *      (custom_all_reduce)", Technical Details, 2stage, reduce-scatter: the
 *      sum of every 16-byte pack is taken in fp32 over the ranks, always in
 *      the order of the pointer array, so it comes out the same bits.
 *   2. two-stage only: t = bf16_rne(acc) and acc := f32(t).  Same section:
 *      stage 1 rounds the sum to bf16 before storing it in the temporary
 *      buffer that stage 2 (local_device_load_rmsnorm) loads.
 *   3. r = acc + f32(residual[i,j]) in fp32; residual_out = bf16_rne(r).
 *      The residual enters after all n partials (AllReduce, then residual add).
 *   4. RMSNorm, as named by the title of aiter #3817 and by its stage-2 section
 *      on the RMSNorm's sum of squares, in its textbook form:
 *      ss = sum_j r_j^2, inv = 1/sqrt(ss/H + eps), out = bf16_rne(r_j*inv*w_j).
 *      The pages fix no precision for this part, so it runs in fp64; only
 *      the final value is rounded (once) to bf16.
 *
 * bf16 values travel as raw 16-bit patterns (uint16_t).
 *
 * Build flags matter: -ffp-contract=off keeps the compiler from fusing a
 * multiply and an add into one rounding (aarch64 gcc would do that by
 * default), so x86_64 and aarch64 builds give the same bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_N 64

/* bf16 -> fp32: a bf16 pattern is the top half of an fp32 pattern. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/*
 * Round a double to the nearest bf16 (ties to even), in one rounding step.
 * bf16 keeps 8 significant bits; normal exponents run from -126 to 127, and
 * below 2^-126 the spacing stays 2^-133 (subnormals).  The value is scaled
 * by a power of two so that the kept bits form an integer, rounded with
 * nearbyint (round-half-even in the default rounding mode), and scaled back;
 * both scalings are exact.  Results above the largest finite bf16
 * ((2 - 2^-7) * 2^127) become infinity.  NaN becomes the quiet NaN 0x7FC0
 * with the input's sign.  Every fp32 is a double, so this also serves as
 * the fp32 -> bf16 conversion.
 */
uint16_t oracle_bf16_from_f64(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0u);
    double ax = fabs(x);
    if (isinf(ax))
        return (uint16_t)(sign | 0x7F80u);
    if (ax == 0.0)
        return sign;
    int e;
    (void)frexp(ax, &e);              /* ax = f * 2^e with f in [0.5, 1) */
    int lead = e - 1;                 /* exponent of the leading bit */
    int qexp = (lead >= -126 ? lead : -126) - 7;
    double y = ldexp(nearbyint(ldexp(ax, -qexp)), qexp);
    if (y > 0x1.FEp127)
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)y;               /* exact: y has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* Step 1 (and 2): the reduced sum of one element, in rank order. */
static float reduce_in_rank_order(const uint16_t *const *partials, int n,
                                  int64_t idx, int two_stage)
{
    float acc = oracle_bf16_to_f32(partials[0][idx]);
    for (int k = 1; k < n; ++k)
        acc = acc + oracle_bf16_to_f32(partials[k][idx]);
    if (two_stage)
        acc = oracle_bf16_to_f32(oracle_bf16_from_f64((double)acc));
    return acc;
}

/*
 * One row.  `r_scratch` holds H floats.  `sum` (may be NULL) receives
 * the reduced sum: the fp32 acc for one-stage, f32(t) for two-stage.
 */
static void oracle_row(const uint16_t *const *partials, int n,
                       const uint16_t *residual, const uint16_t *weight,
                       double eps, int64_t i, int64_t H, int two_stage,
                       uint16_t *out, uint16_t *residual_out, float *sum,
                       float *r_scratch)
{
    const int64_t base = i * H;
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j) {
        float acc = reduce_in_rank_order(partials, n, base + j, two_stage);
        if (sum)
            sum[base + j] = acc;
        float r = acc + oracle_bf16_to_f32(residual[base + j]);
        residual_out[base + j] = oracle_bf16_from_f64((double)r);
        r_scratch[j] = r;
        ss += (double)r * (double)r;
    }
    double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t j = 0; j < H; ++j) {
        double y = (double)r_scratch[j] * inv * (double)oracle_bf16_to_f32(weight[j]);
        out[base + j] = oracle_bf16_from_f64(y);
    }
}

struct oracle_job {
    const uint16_t *const *partials;
    int n;
    const uint16_t *residual, *weight;
    double eps;
    int64_t row_begin, row_end, H;
    int two_stage;
    uint16_t *out, *residual_out;
    float *sum;
    int status;
};

static void *oracle_rows(void *arg)
{
    struct oracle_job *job = (struct oracle_job *)arg;
    float *r = (float *)malloc(sizeof(float) * (size_t)(job->H > 0 ? job->H : 1));
    if (!r) {
        job->status = -2;
        return NULL;
    }
    for (int64_t i = job->row_begin; i < job->row_end; ++i)
        oracle_row(job->partials, job->n, job->residual, job->weight, job->eps,
                   i, job->H, job->two_stage, job->out, job->residual_out,
                   job->sum, r);
    free(r);
    job->status = 0;
    return NULL;
}

/*
 * The whole epilogue over m rows.  All buffers are row-major [m, H] bf16
 * patterns except `weight` ([H]) and `sum` (fp32 [m, H], may be NULL).
 * `threads` > 1 splits the rows into contiguous blocks, one per thread;
 * rows are independent, so the result does not depend on it.
 * Returns 0, -1 for bad arguments, -2 when memory or threads run out.
 */
int oracle_ar_rmsnorm(const uint16_t *const *partials, int n,
                      const uint16_t *residual, const uint16_t *weight,
                      double eps, int64_t m, int64_t H, int two_stage,
                      uint16_t *out, uint16_t *residual_out, float *sum,
                      int threads)
{
    if (n < 1 || n > ORACLE_MAX_N || m < 0 || H < 1 || !partials || !residual
        || !weight || !out || !residual_out)
        return -1;
    for (int k = 0; k < n; ++k)
        if (!partials[k])
            return -1;
    if (threads < 1)
        threads = 1;
    if (threads > m)
        threads = (int)(m > 0 ? m : 1);

    struct oracle_job *jobs = (struct oracle_job *)calloc((size_t)threads, sizeof *jobs);
    pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof *tids);
    char *created = (char *)calloc((size_t)threads, 1);
    if (!jobs || !tids || !created) {
        free(jobs);
        free(tids);
        free(created);
        return -2;
    }
    int64_t per = (m + threads - 1) / threads;
    int status = 0;
    for (int t = 0; t < threads; ++t) {
        struct oracle_job *j = &jobs[t];
        j->partials = partials;
        j->n = n;
        j->residual = residual;
        j->weight = weight;
        j->eps = eps;
        j->row_begin = t * per < m ? t * per : m;
        j->row_end = (t + 1) * per < m ? (t + 1) * per : m;
        j->H = H;
        j->two_stage = two_stage;
        j->out = out;
        j->residual_out = residual_out;
        j->sum = sum;
        j->status = -2;
        if (threads == 1) {
            oracle_rows(j);
        } else if (pthread_create(&tids[t], NULL, oracle_rows, j) == 0) {
            created[t] = 1;
        } else {
            oracle_rows(j); /* run it here if no thread can be had */
        }
    }
    for (int t = 0; t < threads; ++t)
        if (created[t])
            pthread_join(tids[t], NULL);
    for (int t = 0; t < threads; ++t)
        if (jobs[t].status != 0)
            status = jobs[t].status;
    free(jobs);
    free(tids);
    free(created);
    return status;
}
