/*
 * Plain double-precision CPU oracle for the scaled dot-product attention
 * forward pass and its log-sum-exp side output.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker that the CUDA path is
 * compared against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header or constant with
 * the CUDA library and includes nothing from it.
 *
 * Sources (cited by page title and section):
 *   [QS] "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程" (blog.qingsen.net)
 *   [PW] "Flash Attention 前向 ... CUTLASS" (pwwt.cn news repost)
 *   [YT] "CUDA 算子工程" ch. 14 "Attention 的访存瓶颈与 IO-Aware 思想"
 *        (yangyitao.com)
 *
 * What is computed (the plain definition, [QS] section "先固定一个例子",
 * equation S = QK^T, P = softmax_row(sS), O = PV; [YT] section 14.1):
 *   for every batch b, head h and query row i,
 *     x_j   = sum_c q[i][c] * k[j][c]          over the valid keys j
 *     m     = max_j x_j                         (raw, unscaled scores)
 *     l     = sum_j exp(s * (x_j - m))
 *     O[i]  = sum_j exp(s * (x_j - m)) * v[j] / l
 *     LSE_i = s * m + ln(l)                     ([QS] section "最后：归一化并写回 O")
 *   With Nq queries and Nk keys per head, key j is valid when j < Nk and, for
 *   the causal variant, j <= i + offset: offset 0 is the top-left alignment of
 *   [QS] section "causal 模式在哪一步生效", Fig. 11 (whose worked example has 2
 *   queries and 4 keys); offset Nk - Nq is the bottom-right alignment that
 *   section mentions without defining, read here as "the last query sees
 *   every key".  Mask modes: 0 none, 1 top-left, 2 bottom-right.  A row with
 *   no valid key gets O = 0 and LSE = -inf (the pages leave this case open).
 *
 * Subtracting the row maximum before exponentiating is the numerically stable
 * softmax of [PW] section 3.1; it does not change the value.
 *
 * A second routine, oracle_blocked_head(), follows the online-softmax
 * recurrence step by step ([QS] section "第四步：更新 online softmax",
 * Table 2 and the equations for m', alpha, l', U'; [YT] section 14.5), so that
 * the recurrence itself can be checked against the plain definition and
 * against the worked example's printed intermediates.  It is never used to
 * produce expected values for the CUDA path.
 *
 * 16-bit inputs are widened to double exactly, decoding the IEEE binary16 and
 * bfloat16 bit patterns from their definitions.
 *
 * Parity pins: every function here is pinned by tests/test_oracle.py (worked
 * example, causal closed form, invariants, special cases, brute force in
 * arbitrary precision, library log-sum-exp).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FP16 0
#define ORACLE_BF16 1

/* ---- exact widening of 16-bit floating-point bit patterns ---------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_binary16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(frac + 1024), expo - 25);  /* (1 + frac/2^10) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double decode_bfloat16(uint16_t b) {
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 0xff;
    int frac = b & 0x7f;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -133);                /* subnormal: frac * 2^-133 */
    } else if (expo == 255) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(frac + 128), expo - 134);  /* (1 + frac/2^7) * 2^(e-127) */
    }
    return sign ? -mag : mag;
}

void oracle_decode16(const uint16_t* src, int dtype, double* dst, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        dst[i] = dtype == ORACLE_BF16 ? decode_bfloat16(src[i]) : decode_binary16(src[i]);
}

/* ---- one query row, plain definition -------------------------------------- */

/* Keys visible to query row i (a prefix 0 .. result-1 of the Nk keys). */
static int64_t visible_keys(int mask, int64_t i, int64_t Nq, int64_t Nk) {
    if (mask == 0) return Nk;
    int64_t end = i + 1 + (mask == 2 ? Nk - Nq : 0);
    if (end > Nk) end = Nk;
    return end < 0 ? 0 : end;
}

/*
 * q: [d]; k, v: [Nk, d] of one (b, h); the first nvalid keys are visible;
 * x: scratch of Nk doubles.
 * spread (optional, [d]): sum_j P_ij |v_jc - O_ic|, the probability-weighted
 * spread of the values around the output.  It bounds how far O moves when
 * every weight is perturbed by a relative error of at most u: the change in
 * O_ic is at most 2u * spread_c / (1 - u).  Test tolerances use it for the
 * rounding of the weights to 16 bits before the P.V product.
 */
static void attend_row(const double* q, const double* k, const double* v,
                       int64_t nvalid, int64_t d, double s,
                       double* x, double* o_row, double* lse_out, double* spread) {
    if (nvalid <= 0) {
        for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
        if (spread)
            for (int64_t c = 0; c < d; ++c) spread[c] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    /* raw scores x_j = q . k_j */
    for (int64_t j = 0; j < nvalid; ++j) {
        double acc = 0.0;
        const double* kj = k + j * d;
        for (int64_t c = 0; c < d; ++c) acc += q[c] * kj[c];
        x[j] = acc;
    }
    /* row maximum of the raw scores */
    double m = x[0];
    for (int64_t j = 1; j < nvalid; ++j)
        if (x[j] > m) m = x[j];
    /* weights relative to m, their sum, and the weighted sum of values */
    double l = 0.0;
    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    for (int64_t j = 0; j < nvalid; ++j) {
        double w = exp(s * (x[j] - m));
        l += w;
        const double* vj = v + j * d;
        for (int64_t c = 0; c < d; ++c) o_row[c] += w * vj[c];
    }
    for (int64_t c = 0; c < d; ++c) o_row[c] /= l;
    *lse_out = s * m + log(l);
    if (spread) {
        for (int64_t c = 0; c < d; ++c) spread[c] = 0.0;
        for (int64_t j = 0; j < nvalid; ++j) {
            double p = exp(s * (x[j] - m)) / l;
            const double* vj = v + j * d;
            for (int64_t c = 0; c < d; ++c) spread[c] += p * fabs(vj[c] - o_row[c]);
        }
    }
}

/* ---- double inputs, whole tensors ----------------------------------------- */

/* q, o: [BH, Nq, d]; k, v: [BH, Nk, d] doubles; lse: [BH, Nq]; mask 0/1/2.
 * Single-threaded. */
int oracle_attention_f64(const double* q, const double* k, const double* v,
                         int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                         double scale, int causal, double* o, double* lse) {
    if (BH < 0 || Nq < 0 || Nk < 0 || d <= 0) return 1;
    double* x = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    if (!x) return 2;
    for (int64_t bh = 0; bh < BH; ++bh) {
        const double* qh = q + bh * Nq * d;
        const double* kh = k + bh * Nk * d;
        const double* vh = v + bh * Nk * d;
        for (int64_t i = 0; i < Nq; ++i)
            attend_row(qh + i * d, kh, vh, visible_keys(causal, i, Nq, Nk), d, scale, x,
                       o + (bh * Nq + i) * d, lse + bh * Nq + i, NULL);
    }
    free(x);
    return 0;
}

/* ---- 16-bit inputs, selected rows, multi-threaded -------------------------- */

typedef struct {
    const uint16_t *q, *k, *v;
    int dtype;
    int64_t Nq, Nk, d;
    double scale;
    int causal;            /* mask mode 0/1/2 */
    const int64_t* rows;   /* flat indices bh * Nq + i, sorted by bh for reuse */
    int64_t nrows;
    double* o;             /* [nrows, d] */
    double* lse;           /* [nrows] */
    double* spread;        /* [nrows, d] or NULL */
    int64_t next;          /* work counter (rows handed out in chunks) */
    pthread_mutex_t lock;
    int failed;
} rows_job_t;

#define ROWS_CHUNK 16

static void* rows_worker(void* arg) {
    rows_job_t* job = (rows_job_t*)arg;
    const int64_t Nq = job->Nq, Nk = job->Nk, d = job->d;
    double* kh = (double*)malloc(sizeof(double) * (size_t)(Nk * d + 1));
    double* vh = (double*)malloc(sizeof(double) * (size_t)(Nk * d + 1));
    double* qr = (double*)malloc(sizeof(double) * (size_t)d);
    double* x = (double*)malloc(sizeof(double) * (size_t)(Nk + 1));
    if (!kh || !vh || !qr || !x) {
        pthread_mutex_lock(&job->lock);
        job->failed = 1;
        pthread_mutex_unlock(&job->lock);
        free(kh); free(vh); free(qr); free(x);
        return NULL;
    }
    int64_t cached_bh = -1;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t start = job->next;
        job->next += ROWS_CHUNK;
        pthread_mutex_unlock(&job->lock);
        if (start >= job->nrows) break;
        int64_t end = start + ROWS_CHUNK < job->nrows ? start + ROWS_CHUNK : job->nrows;
        for (int64_t r = start; r < end; ++r) {
            int64_t flat = job->rows[r];
            int64_t bh = flat / Nq, i = flat % Nq;
            if (bh != cached_bh) {
                oracle_decode16(job->k + bh * Nk * d, job->dtype, kh, Nk * d);
                oracle_decode16(job->v + bh * Nk * d, job->dtype, vh, Nk * d);
                cached_bh = bh;
            }
            oracle_decode16(job->q + flat * d, job->dtype, qr, d);
            attend_row(qr, kh, vh, visible_keys(job->causal, i, Nq, Nk), d, job->scale, x,
                       job->o + r * d, job->lse + r,
                       job->spread ? job->spread + r * d : NULL);
        }
    }
    free(kh); free(vh); free(qr); free(x);
    return NULL;
}

/*
 * q: [BH, Nq, d], k, v: [BH, Nk, d] raw 16-bit patterns of `dtype`; mask
 * mode 0/1/2.  rows: nrows flat row indices (bh * Nq + i), each in
 * [0, BH * Nq).  o: [nrows, d], lse: [nrows], spread: [nrows, d] or NULL (see
 * attend_row).  Returns 0 on success.
 */
int oracle_attention_rows16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            int dtype, int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                            double scale, int causal,
                            const int64_t* rows, int64_t nrows,
                            double* o, double* lse, double* spread, int nthreads) {
    if (BH <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || nrows < 0) return 1;
    if (dtype != ORACLE_FP16 && dtype != ORACLE_BF16) return 1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= BH * Nq) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    rows_job_t job;
    job.q = q; job.k = k; job.v = v; job.dtype = dtype;
    job.Nq = Nq; job.Nk = Nk; job.d = d; job.scale = scale; job.causal = causal;
    job.rows = rows; job.nrows = nrows; job.o = o; job.lse = lse; job.spread = spread;
    job.next = 0; job.failed = 0;
    pthread_mutex_init(&job.lock, NULL);
    pthread_t tids[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, rows_worker, &job) != 0) break;
        ++started;
    }
    if (started == 0) rows_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.failed ? 2 : 0;
}

/* ---- the online-softmax recurrence, literally, for one head ---------------- */

/*
 * Walks the keys in blocks of block_n and keeps, per query row, the running
 * maximum m of the raw scores, the sum l of the weights relative to m, and
 * the unnormalised output numerator U ([QS] section "第四步", Table 2):
 *   first block with a valid key:  m = max_B x,  l = sum_B e^{s(x-m)},
 *                                  U = sum_B e^{s(x-m)} v        (no rescale)
 *   later blocks:  m' = max(m, max_B x),  alpha = e^{s(m - m')},
 *                  l' = alpha l + sum_B e^{s(x - m')},
 *                  U' = alpha U + sum_B e^{s(x - m')} v
 *   at the end:    O = U / l,  LSE = s m + ln l   ([QS] section "最后")
 * Blocks without a valid key are skipped, as the causal variant skips tiles
 * that lie wholly in the future.
 *
 * q, o: [Nq, d]; k, v: [Nk, d]; lse: [Nq].  The optional trace arrays, indexed
 * by block t (nblk = ceil(Nk / block_n)), record the state after each block:
 *   trace_m[t*Nq + i], trace_l[t*Nq + i], trace_alpha[t*Nq + i] (NaN for the
 *   first valid block and for skipped blocks), trace_u[(t*Nq + i)*d + c],
 *   trace_e[(t*Nq + i)*block_n + jj] (weights of the block's keys; 0 if masked).
 * Any trace pointer may be NULL.
 */
int oracle_blocked_head(const double* q, const double* k, const double* v,
                        int64_t Nq, int64_t Nk, int64_t d, double scale, int causal,
                        int64_t block_n,
                        double* o, double* lse,
                        double* trace_m, double* trace_l, double* trace_alpha,
                        double* trace_u, double* trace_e) {
    if (Nq < 0 || Nk < 0 || d <= 0 || block_n <= 0) return 1;
    int64_t nblk = (Nk + block_n - 1) / block_n;
    double* x = (double*)malloc(sizeof(double) * (size_t)block_n);
    double* u = (double*)malloc(sizeof(double) * (size_t)d);
    if (!x || !u) { free(x); free(u); return 2; }
    for (int64_t i = 0; i < Nq; ++i) {
        const double* qi = q + i * d;
        int have_state = 0;
        double m = -INFINITY, l = 0.0;
        for (int64_t c = 0; c < d; ++c) u[c] = 0.0;
        for (int64_t t = 0; t < nblk; ++t) {
            int64_t j0 = t * block_n;
            int64_t j1 = j0 + block_n < Nk ? j0 + block_n : Nk;
            /* valid keys of this block */
            int64_t jend = j1;
            const int64_t vis = visible_keys(causal, i, Nq, Nk);
            if (vis < jend) jend = vis;
            double alpha = NAN;
            if (trace_e)
                for (int64_t jj = 0; jj < block_n; ++jj) trace_e[(t * Nq + i) * block_n + jj] = 0.0;
            if (jend > j0) {
                double mb = -INFINITY;
                for (int64_t j = j0; j < jend; ++j) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; ++c) acc += qi[c] * k[j * d + c];
                    x[j - j0] = acc;
                    if (acc > mb) mb = acc;
                }
                double m_new = have_state ? (m > mb ? m : mb) : mb;
                if (have_state) {
                    alpha = exp(scale * (m - m_new));
                    l *= alpha;
                    for (int64_t c = 0; c < d; ++c) u[c] *= alpha;
                }
                for (int64_t j = j0; j < jend; ++j) {
                    double w = exp(scale * (x[j - j0] - m_new));
                    if (trace_e) trace_e[(t * Nq + i) * block_n + (j - j0)] = w;
                    l += w;
                    for (int64_t c = 0; c < d; ++c) u[c] += w * v[j * d + c];
                }
                m = m_new;
                have_state = 1;
            }
            if (trace_m) trace_m[t * Nq + i] = m;
            if (trace_l) trace_l[t * Nq + i] = l;
            if (trace_alpha) trace_alpha[t * Nq + i] = alpha;
            if (trace_u)
                for (int64_t c = 0; c < d; ++c) trace_u[(t * Nq + i) * d + c] = u[c];
        }
        if (!have_state) {
            for (int64_t c = 0; c < d; ++c) o[i * d + c] = 0.0;
            lse[i] = -INFINITY;
        } else {
            for (int64_t c = 0; c < d; ++c) o[i * d + c] = u[c] / l;
            lse[i] = scale * m + log(l);
        }
    }
    free(x);
    free(u);
    return 0;
}

int oracle_version(void) { return 1; }
