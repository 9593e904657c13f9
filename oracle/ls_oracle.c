/*
 * ls_oracle.c -- plain, slow, double-precision CPU oracle for the per-token
 * decode step of delta-rule linear attention over a pool of recurrent states.
 *
 * TEST INFRASTRUCTURE ONLY.  It is called by the test-suite, by the smoke
 * check and by the CPU-baseline leg of the benchmark; the product (the CUDA
 * library and its Python binding) never loads it.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * Sources (page title, then section / equation / algorithm):
 *   [LQ] "LeapQuant: Efficient Linear Attention with Accurate Recurrent State
 *        Quantization" (arXiv 2609.38166).
 *   [DL] "DeltaLog: Deferred Materialization of Recurrent States for Linear
 *        Attention Decoding" (arXiv 2608.15533).
 *
 * Conventions
 *   One head's state S is d_k x d_v, stored row-major: S[i*dv + j], i = key
 *   row, j = value column.  All state arithmetic is in double.
 *   The gate arrives as a log-decay lambda <= 0 ([DL] §2.1 eq. 2-3):
 *   alpha = exp(lambda).  dl == 1 is the scalar gate of Gated DeltaNet (one
 *   lambda per head and token), dl == dk the per-key gate of KDA.
 *   Every batched entry point takes n rows; row r reads its own inputs
 *   (q[r*dk..], k[r*dk..], v[r*dv..], lam[r*dl..], beta[r]) and updates the
 *   state with index idx[r] of a state array.  Rows must name distinct states.
 *
 * Readings of points the pages leave open (each one is listed in the design
 * notes of the repository):
 *   - beta sits in the correction: u = beta (v - S^T (alpha . k))
 *     ([LQ] App. A, GDN and KDA rows and the remark that follows them).
 *   - The delta-rule readout uses the decayed state, S^T (alpha . k), as in
 *     the right-hand sides of [LQ] App. A.
 *   - The output is always the post-update readout y = S_t^T q_t ([LQ] eq. 1).
 *   - INT8 per-window scheme: symmetric INT8 with one FP32 scale per key row:
 *     B_i = max_j |S_ij|, Z = clamp(round-half-even(S * (127 / B_i)), -127, 127),
 *     stored scale s_i = B_i / 127 ([LQ] App. B.3 writes dequant = (Z/127) B);
 *     a zero row (or one whose factor overflows) gets s = 0 and Z = 0.  The
 *     decision (absmax, factor, product, rounding) is taken in FP32 on the
 *     FP32 rounding of the double state, the precision the CUDA kernel
 *     computes in.
 *   - The window counts tokens from the last boundary (load, commit or
 *     reset); the W-th token's output is read from the unquantized S_W, then
 *     S_W is quantized ([LQ] §3.2 eq. 4).  W = 1 is per-step quantization
 *     ([LQ] §3.2 eq. 2).
 *   - Deferred cycle: merge interval M, live-log capacity C = M - 1
 *     ([DL] §3.1).  M = 1 merges at every token, i.e. eager decoding.
 *   - An explicit commit of a state with an empty log/window leaves it as it
 *     is (nothing to fold, the state is already at a boundary).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_NOMEM -2

static int valid_dims(int dk, int dv, int dl)
{
    return dk > 0 && dv > 0 && (dl == 1 || dl == dk);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* lambda of key row i (scalar gate: the same value for every row). */
static double lam_at(const float *lam, int dl, int i)
{
    return (double)lam[dl == 1 ? 0 : i];
}

static double dlam_at(const double *lam, int dl, int i)
{
    return lam[dl == 1 ? 0 : i];
}

/* ------------------------------------------------------------------------ */
/* Eager recurrence                                                          */
/* ------------------------------------------------------------------------ */

/*
 * One token on one head, straight from the definition.
 * [LQ] App. A (GDN / KDA rows, right-hand side) together with [LQ] eq. 1:
 *     w   = alpha . k
 *     r   = S_{t-1}^T w
 *     u   = beta (v - r)
 *     S_t = Diag(alpha) S_{t-1} + k u^T
 *     y   = S_t^T q
 * y is formed from the updated S_t itself, not from a fused expression.
 * u_out (dv doubles) receives u when non-NULL.
 * rule 1 (no delta correction): u = v, the update pair (k_t, v_t) of the
 * linear attention / RetNet / GLA / RWKV6 rows of [DL] Table 1 (read vector
 * b_t = 0 in [LQ] App. A); beta is not used.
 */
static void eager_one(int rule, int dk, int dv, int dl, double *S,
                      const float *q, const float *k, const float *v,
                      const float *lam, float beta, double *y, double *r,
                      double *u_out)
{
    for (int j = 0; j < dv; ++j) r[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
        const double w = exp(lam_at(lam, dl, i)) * (double)k[i];
        const double *Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) r[j] += Si[j] * w;
    }
    /* u overwrites r in place */
    for (int j = 0; j < dv; ++j)
        r[j] = rule == 1 ? (double)v[j] : (double)beta * ((double)v[j] - r[j]);
    for (int i = 0; i < dk; ++i) {
        const double a = exp(lam_at(lam, dl, i));
        const double ki = (double)k[i];
        double *Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) Si[j] = a * Si[j] + ki * r[j];
    }
    for (int j = 0; j < dv; ++j) y[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
        const double qi = (double)q[i];
        const double *Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) y[j] += Si[j] * qi;
    }
    if (u_out)
        for (int j = 0; j < dv; ++j) u_out[j] = r[j];
}

int orc_eager_step(int64_t n, int rule, int dk, int dv, int dl, double *S,
                   const int64_t *idx, const float *q, const float *k,
                   const float *v, const float *lam, const float *beta,
                   double *y, int nthreads)
{
    if (n < 0 || !valid_dims(dk, dv, dl) || (rule != 0 && rule != 1)) return ORC_ERR_ARG;
    if (n == 0) return ORC_OK;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *r = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!r) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t row = 0; row < n; ++row) {
                double *Sr = S + (size_t)idx[row] * dk * dv;
                eager_one(rule, dk, dv, dl, Sr, q + row * dk, k + row * dk,
                          v + row * dv, lam + row * dl, beta[row],
                          y + row * dv, r, NULL);
            }
        }
        free(r);
    }
    return err ? ORC_ERR_NOMEM : ORC_OK;
}

/*
 * 16-bit key-side log factors ([DL] §3.4: "deferred key-side factors a_t
 * use 16-bit storage" for GDN and KDA): k stored as bfloat16, the FP32 value
 * rounded to its top 16 bits, round half to even on the discarded bits.
 */
static double bf16_round(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    const uint32_t lsb = (b >> 16) & 1u;
    b = (b + 0x7fffu + lsb) & 0xffff0000u;
    float y;
    memcpy(&y, &b, 4);
    return (double)y;
}

/*
 * FP16 records ([LQ] §4.3: the window's buffered records and the r
 * compensator pairs are kept in FP16): x rounded to the nearest IEEE
 * binary16 number, ties to even.  In [2^(e-1), 2^e) binary16 has 11
 * significant bits, so its spacing is 2^(e-11); below 2^-14 (subnormals)
 * the spacing stays 2^-24.  A magnitude that rounds above 65504 is infinite.
 */
static double fp16_round(double x)
{
    if (x == 0.0 || isnan(x) || isinf(x)) return x;
    const double a = fabs(x);
    int e;
    (void)frexp(a, &e); /* 2^(e-1) <= a < 2^e */
    int q = e - 11;
    if (q < -24) q = -24;
    const double step = ldexp(1.0, q);
    double r = rint(a / step) * step; /* a / step is exact */
    if (r > 65504.0) r = INFINITY;
    return copysign(r, x);
}

/* Record formats: 0 FP32; 1 bfloat16 keys ([DL] §3.4); 2 FP16 keys and
 * values, and FP16 compensator pairs ([LQ] §4.3). */
#define REC_FP32 0
#define REC_BF16_K 1
#define REC_FP16 2

static double stored_key(int rec, float k)
{
    if (rec == REC_BF16_K) return bf16_round(k);
    if (rec == REC_FP16) return fp16_round((double)k);
    return (double)k;
}

/* ------------------------------------------------------------------------ */
/* Deferred materialization (base + bounded log)                             */
/* ------------------------------------------------------------------------ */

/*
 * Per-state arrays of the deferred representation ([DL] §3.1):
 *   base  [dk*dv]   dense base state S-bar
 *   lbar  [dl]      cumulative log-decay since the last materialization
 *   K     [C*dk]    key-side factors  K_log
 *   U     [C*dv]    value-side factors U_log
 *   Lam   [C*dl]    log-decay snapshot Lambda_log of every entry
 *   L               live-log length, 0 <= L <= C = M - 1
 */

/*
 * Logical state represented by base + log, [DL] §3.2 eq. 7:
 *   S = D(lbar) S-bar + sum_{l<L} D(lbar - Lambda_l) K_l U_l^T,
 * with D(x) = diag(exp(x)) ([DL] eq. 2).  `lb` is the cumulative log-decay
 * to use (the stored one, or the one after the current token's lambda).
 */
static void deferred_represented(int dk, int dv, int dl, const double *base,
                                 const double *lb, const double *K,
                                 const double *U, const double *Lam, int L,
                                 double *S)
{
    for (int i = 0; i < dk; ++i) {
        const double e = exp(dlam_at(lb, dl, i));
        for (int j = 0; j < dv; ++j)
            S[(size_t)i * dv + j] = e * base[(size_t)i * dv + j];
    }
    for (int l = 0; l < L; ++l) {
        const double *Kl = K + (size_t)l * dk;
        const double *Ul = U + (size_t)l * dv;
        const double *Ll = Lam + (size_t)l * dl;
        for (int i = 0; i < dk; ++i) {
            const double g = exp(dlam_at(lb, dl, i) - dlam_at(Ll, dl, i));
            const double a = g * Kl[i];
            double *Si = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) Si[j] += a * Ul[j];
        }
    }
}

/*
 * One token on one deferred state, [DL] §3.1 Algorithm 1 with eq. 4-6:
 *   1. pre-update readout of the old logical state (eq. 7):
 *        r = S_{t-1}^T (alpha . k)
 *   2. lbar <- lbar + lambda_t                                   (eq. 4)
 *   3. update factors a_t = k, b_t = u = beta (v - r); the post-update
 *      output y = S_t^T q with S_t the logical state that includes the
 *      current update
 *   4. L < C : append (k, u, lbar) at entry L, L <- L + 1       (eq. 5)
 *      L = C : S-bar <- D(lbar) S-bar + sum D(lbar - Lambda_i) K_i U_i^T
 *                       + a_t b_t^T, then lbar <- 0, L <- 0     (eq. 6)
 * work: 2*dk*dv doubles.  rule 1: b_t = v (no delta correction, as eager_one).
 * k16: the appended key-side factor is bf16(k) ([DL] §3.4); the token's own
 * output and a merge that folds it use k itself.
 */
static void deferred_one(int rule, int k16, int dk, int dv, int dl, int M, double *base,
                         double *lbar, double *K, double *U, double *Lam,
                         int32_t *Lp, const float *q, const float *k,
                         const float *v, const float *lam, float beta,
                         double *y, double *work)
{
    const int C = M - 1;
    const int L = *Lp;
    double *Sprev = work;
    double *St = work + (size_t)dk * dv;
    double r[1024];
    double lnew[1024];

    /* 1. readout from the pre-update logical state */
    deferred_represented(dk, dv, dl, base, lbar, K, U, Lam, L, Sprev);
    for (int j = 0; j < dv; ++j) r[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
        const double w = exp(lam_at(lam, dl, i)) * (double)k[i];
        for (int j = 0; j < dv; ++j) r[j] += Sprev[(size_t)i * dv + j] * w;
    }
    /* 2. cumulative log-decay */
    lnew[0] = 0.0;
    for (int c = 0; c < dl; ++c) lnew[c] = lbar[c] + (double)lam[c];
    /* 3. update factors and post-update output */
    double u[1024];
    for (int j = 0; j < dv; ++j)
        u[j] = rule == 1 ? (double)v[j] : (double)beta * ((double)v[j] - r[j]);
    deferred_represented(dk, dv, dl, base, lnew, K, U, Lam, L, St);
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            St[(size_t)i * dv + j] += (double)k[i] * u[j];
    for (int j = 0; j < dv; ++j) y[j] = 0.0;
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            y[j] += St[(size_t)i * dv + j] * (double)q[i];
    /* 4. append or merge */
    if (L < C) {
        for (int i = 0; i < dk; ++i) K[(size_t)L * dk + i] = stored_key(k16, k[i]);
        for (int j = 0; j < dv; ++j) U[(size_t)L * dv + j] = u[j];
        for (int c = 0; c < dl; ++c) Lam[(size_t)L * dl + c] = lnew[c];
        for (int c = 0; c < dl; ++c) lbar[c] = lnew[c];
        *Lp = L + 1;
    } else {
        memcpy(base, St, sizeof(double) * (size_t)dk * dv);
        for (int c = 0; c < dl; ++c) lbar[c] = 0.0;
        *Lp = 0;
    }
}

static int deferred_args_ok(int dk, int dv, int dl, int M)
{
    return valid_dims(dk, dv, dl) && M >= 1 && dk <= 1024 && dv <= 1024;
}

int orc_deferred_step(int64_t n, int rule, int k16, int dk, int dv, int dl, int M,
                      double *base, double *lbar, double *K, double *U,
                      double *Lam, int32_t *L, const int64_t *idx,
                      const float *q, const float *k, const float *v,
                      const float *lam, const float *beta, double *y,
                      int nthreads)
{
    if (n < 0 || !deferred_args_ok(dk, dv, dl, M) || (rule != 0 && rule != 1))
        return ORC_ERR_ARG;
    if (n == 0) return ORC_OK;
    const int C = M - 1;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *work = (double *)malloc(sizeof(double) * 2 * (size_t)dk * dv);
        if (!work) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 2)
            for (int64_t row = 0; row < n; ++row) {
                const int64_t s = idx[row];
                deferred_one(rule, k16, dk, dv, dl, M, base + (size_t)s * dk * dv,
                             lbar + (size_t)s * dl, K + (size_t)s * C * dk,
                             U + (size_t)s * C * dv, Lam + (size_t)s * C * dl,
                             L + s, q + row * dk, k + row * dk, v + row * dv,
                             lam + row * dl, beta[row], y + row * dv, work);
            }
        }
        free(work);
    }
    return err ? ORC_ERR_NOMEM : ORC_OK;
}

/* Logical state of n deferred states ([DL] eq. 7), without changing them. */
int orc_deferred_logical(int64_t n, int dk, int dv, int dl, int M,
                         const double *base, const double *lbar,
                         const double *K, const double *U, const double *Lam,
                         const int32_t *L, const int64_t *idx, double *S_out)
{
    if (n < 0 || !deferred_args_ok(dk, dv, dl, M)) return ORC_ERR_ARG;
    const int C = M - 1;
#pragma omp parallel for schedule(dynamic, 2)
    for (int64_t row = 0; row < n; ++row) {
        const int64_t s = idx[row];
        deferred_represented(dk, dv, dl, base + (size_t)s * dk * dv,
                             lbar + (size_t)s * dl, K + (size_t)s * C * dk,
                             U + (size_t)s * C * dv, Lam + (size_t)s * C * dl,
                             L[s], S_out + (size_t)row * dk * dv);
    }
    return ORC_OK;
}

/*
 * Explicit merge with no new token: materialize eq. 7 into the base, then
 * reset lbar and L, as the merge branch of [DL] Algorithm 1 does.  An empty
 * log is left alone.
 */
int orc_deferred_commit(int64_t n, int dk, int dv, int dl, int M,
                        double *base, double *lbar, double *K, double *U,
                        double *Lam, int32_t *L, const int64_t *idx)
{
    if (n < 0 || !deferred_args_ok(dk, dv, dl, M)) return ORC_ERR_ARG;
    const int C = M - 1;
    int err = 0;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
        if (!S) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 2)
            for (int64_t row = 0; row < n; ++row) {
                const int64_t s = idx[row];
                if (L[s] == 0) continue;
                double *b = base + (size_t)s * dk * dv;
                double *lb = lbar + (size_t)s * dl;
                deferred_represented(dk, dv, dl, b, lb, K + (size_t)s * C * dk,
                                     U + (size_t)s * C * dv,
                                     Lam + (size_t)s * C * dl, L[s], S);
                memcpy(b, S, sizeof(double) * (size_t)dk * dv);
                for (int c = 0; c < dl; ++c) lb[c] = 0.0;
                L[s] = 0;
            }
        }
        free(S);
    }
    return err ? ORC_ERR_NOMEM : ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Symmetric INT8 with one FP32 scale per key row                           */
/* ------------------------------------------------------------------------ */

/*
 * quant_8 of [LQ] §3.1 / App. B.3, one scale per key row.  App. B.3 writes
 * the dequantization as (Z / 127) B with B the row's absmax, so the row is
 * quantized by the factor 127 / B:
 *     Z_ij = clamp(round-half-even(S_ij * (127 / B_i)), -127, 127),
 *     stored scale s_i = B_i / 127 (dequant S_ij = s_i Z_ij).
 * The decision is taken in FP32 on the FP32 rounding of S: B_i, 127 / B_i,
 * B_i / 127 and the product are each correctly rounded FP32 operations.  A
 * row whose scale or factor is not a positive finite FP32 number (a zero row,
 * or one so small that 127 / B overflows) gets s = 0 and Z = 0.
 */
static void quant_rows(int dk, int dv, const double *S, int8_t *Z, float *s)
{
    for (int i = 0; i < dk; ++i) {
        float amax = 0.0f;
        for (int j = 0; j < dv; ++j) {
            const float a = fabsf((float)S[(size_t)i * dv + j]);
            if (a > amax) amax = a;
        }
        float sc = amax / 127.0f;
        float inv = amax > 0.0f ? 127.0f / amax : 0.0f;
        if (!(sc > 0.0f) || !(inv <= FLT_MAX)) {
            sc = 0.0f;
            inv = 0.0f;
        }
        s[i] = sc;
        for (int j = 0; j < dv; ++j) {
            int8_t z = 0;
            if (sc > 0.0f) {
                const float x = (float)S[(size_t)i * dv + j];
                float t = rintf(x * inv);
                if (t > 127.0f) t = 127.0f;
                if (t < -127.0f) t = -127.0f;
                z = (int8_t)t;
            }
            Z[(size_t)i * dv + j] = z;
        }
    }
}

/* dequant_8: S_ij = s_i * Z_ij, in double. */
static void dequant_rows(int dk, int dv, const int8_t *Z, const float *s,
                         double *S)
{
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            S[(size_t)i * dv + j] = (double)s[i] * (double)Z[(size_t)i * dv + j];
}

/*
 * The smoothed, per-value-column format of [LQ] §3.4 eq. 7 and App. B.3.
 * The residual (here the whole boundary state) is divided row by row by the
 * smoothing vector c, with c_i the square root of key row i's mean absolute
 * value and a small positive floor, and the result is quantized with one
 * symmetric INT8 scale per value column j: dequant = (Z / 127) B, so
 * S ~ C (Z / 127) B.  Decisions in FP32 on the FP32 rounding of S:
 *     m_i = fl(sum_j |S_ij|) / dv  (sum formed in double, then rounded)
 *     c_i = max(sqrt_fp32(m_i), 2^-20)
 *     g_i = fl(1 / c_i),  R_ij = fl(S_ij * g_i)               (C^-1 S)
 *     B_j = max_i |R_ij|,  b_j = fl(B_j / 127),  f_j = fl(127 / B_j)
 *     Z_ij = round-half-even(fl(R_ij * f_j))
 * A column whose b or f is not a positive finite FP32 number gets b = 0 and
 * Z = 0.  |R_ij f_j| < 127.5, so no clamp acts.  Stored: Z, c (row
 * factors), b (column factors); dequant S_ij = c_i Z_ij b_j.
 */
#define SMOOTH_FLOOR 9.5367431640625e-07f /* 2^-20 */

static void quant_cols(int dk, int dv, const double *S, int8_t *Z, float *c,
                       float *b)
{
    float R[1024];
    float B[1024];
    for (int j = 0; j < dv; ++j) B[j] = 0.0f;
    for (int i = 0; i < dk; ++i) {
        double sum = 0.0;
        for (int j = 0; j < dv; ++j) sum += fabs((double)(float)S[(size_t)i * dv + j]);
        const float m = (float)sum / (float)dv;
        float ci = sqrtf(m);
        if (!(ci >= SMOOTH_FLOOR)) ci = SMOOTH_FLOOR;
        c[i] = ci;
        const float g = 1.0f / ci;
        for (int j = 0; j < dv; ++j) {
            const float r = (float)S[(size_t)i * dv + j] * g;
            const float a = fabsf(r);
            if (a > B[j]) B[j] = a;
        }
    }
    for (int j = 0; j < dv; ++j) {
        float bj = B[j] / 127.0f;
        float fj = B[j] > 0.0f ? 127.0f / B[j] : 0.0f;
        if (!(bj > 0.0f) || !(fj <= FLT_MAX)) {
            bj = 0.0f;
            fj = 0.0f;
        }
        b[j] = bj;
        R[j] = fj;  /* reuse R as the factors */
    }
    for (int i = 0; i < dk; ++i) {
        const float g = 1.0f / c[i];
        for (int j = 0; j < dv; ++j) {
            int8_t z = 0;
            if (b[j] > 0.0f) {
                const float r = (float)S[(size_t)i * dv + j] * g;
                float t = rintf(r * R[j]);
                if (t > 127.0f) t = 127.0f;
                if (t < -127.0f) t = -127.0f;
                z = (int8_t)t;
            }
            Z[(size_t)i * dv + j] = z;
        }
    }
}

/* S_ij = c_i * Z_ij * b_j, in double. */
static void dequant_cols(int dk, int dv, const int8_t *Z, const float *c,
                         const float *b, double *S)
{
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            S[(size_t)i * dv + j] =
                (double)c[i] * (double)Z[(size_t)i * dv + j] * (double)b[j];
}

/* The scheme's two formats: mode 0 = per key row (fr = s, fc unused),
 * mode 1 = smoothed per value column (fr = c, fc = b). */
static void quant_mode(int mode, int dk, int dv, const double *S, int8_t *Z,
                       float *fr, float *fc)
{
    if (mode == 1) quant_cols(dk, dv, S, Z, fr, fc);
    else quant_rows(dk, dv, S, Z, fr);
}

static void dequant_mode(int mode, int dk, int dv, const int8_t *Z,
                         const float *fr, const float *fc, double *S)
{
    if (mode == 1) dequant_cols(dk, dv, Z, fr, fc, S);
    else dequant_rows(dk, dv, Z, fr, S);
}

/*
 * Compensator Tokens, [LQ] §3.3 eq. 5-6: r rank-one pairs (k~_h, u~_h)
 * fitted to the state before quantization, fitted by power iteration (§4.1).
 * Readings (the pages give neither): sequential deflation, h = 1..r, each
 * fit on the residual left by the previous ones; COMP_ITERS power steps
 *     v <- R^T (R v) / ||R^T (R v)||     (v kept if the norm is 0)
 * from the all-ones vector / sqrt(dv) (a warm start from the previous
 * window's pairs can lie in the subspace the earlier pairs just removed,
 * where the steps amplify rounding); then k~_h = R v, u~_h = v (unit),
 * R <- R - k~_h u~_h^T.  With warm != 0 (a test hook) the start is cu[h].
 */
#define COMP_ITERS 3

static void fit_compensators(int r, int dk, int dv, double *R, double *ck,
                             double *cu, int warm, int rec)
{
    double v[1024], z[1024], w[1024];
    for (int h = 0; h < r; ++h) {
        double *u = cu + (size_t)h * dv, *kk = ck + (size_t)h * dk;
        double nv = 0.0;
        if (warm)
            for (int j = 0; j < dv; ++j) nv += u[j] * u[j];
        for (int j = 0; j < dv; ++j)
            v[j] = nv > 0.0 ? u[j] / sqrt(nv) : 1.0 / sqrt((double)dv);
        for (int it = 0; it < COMP_ITERS; ++it) {
            for (int i = 0; i < dk; ++i) {
                double a = 0.0;
                for (int j = 0; j < dv; ++j) a += R[(size_t)i * dv + j] * v[j];
                w[i] = a;
            }
            double nz = 0.0;
            for (int j = 0; j < dv; ++j) {
                double a = 0.0;
                for (int i = 0; i < dk; ++i) a += R[(size_t)i * dv + j] * w[i];
                z[j] = a;
                nz += a * a;
            }
            if (nz > 0.0)
                for (int j = 0; j < dv; ++j) v[j] = z[j] / sqrt(nz);
        }
        for (int i = 0; i < dk; ++i) {
            double a = 0.0;
            for (int j = 0; j < dv; ++j) a += R[(size_t)i * dv + j] * v[j];
            kk[i] = a;
        }
        for (int j = 0; j < dv; ++j) u[j] = v[j];
        /* FP16 pairs: the stored (rounded) pair is the one the residual
         * loses, so the next pair is fitted to what is left of it */
        if (rec == REC_FP16) {
            for (int i = 0; i < dk; ++i) kk[i] = fp16_round(kk[i]);
            for (int j = 0; j < dv; ++j) u[j] = fp16_round(u[j]);
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) R[(size_t)i * dv + j] -= kk[i] * u[j];
    }
}

/* The fit alone, for n states: S [n][dk][dv] in, the residual out; ck, cu
 * [n][r][dk], [n][r][dv] (cu is also the warm start when warm != 0). */
int orc_fit_compensators(int64_t n, int r, int dk, int dv, double *S,
                         double *ck, double *cu, int warm)
{
    if (n < 0 || r < 1 || r > 64 || dk <= 0 || dv <= 0 || dk > 1024 || dv > 1024)
        return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < n; ++h)
        fit_compensators(r, dk, dv, S + (size_t)h * dk * dv, ck + (size_t)h * r * dk,
                         cu + (size_t)h * r * dv, warm, REC_FP32);
    return ORC_OK;
}

/*
 * A window boundary, [LQ] eq. 4 with §3.3 eq. 6 and §3.4 eq. 7: S (the
 * state reached, in place) -> fit r compensator pairs to it, quantize the
 * residual R = S - K~ U~^T in the pool's format, and restart the window
 * from dequant(R-hat) + K~ U~^T.  r = 0: plain quantization of S.
 */
static void boundary(int mode, int r, int rec, int dk, int dv, double *S, int8_t *Z,
                     float *s, float *fc, double *ck, double *cu, int warm)
{
    (void)warm;
    if (r > 0) fit_compensators(r, dk, dv, S, ck, cu, 0, rec);
    quant_mode(mode, dk, dv, S, Z, s, fc);
    dequant_mode(mode, dk, dv, Z, s, fc, S);
    for (int h = 0; h < r; ++h)
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] += ck[(size_t)h * dk + i] * cu[(size_t)h * dv + j];
}

int orc_quantize_rows(int64_t n, int dk, int dv, const double *S, int8_t *Z,
                      float *s)
{
    if (n < 0 || dk <= 0 || dv <= 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < n; ++h)
        quant_rows(dk, dv, S + (size_t)h * dk * dv, Z + (size_t)h * dk * dv,
                   s + (size_t)h * dk);
    return ORC_OK;
}

int orc_dequantize_rows(int64_t n, int dk, int dv, const int8_t *Z,
                        const float *s, double *S)
{
    if (n < 0 || dk <= 0 || dv <= 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < n; ++h)
        dequant_rows(dk, dv, Z + (size_t)h * dk * dv, s + (size_t)h * dk,
                     S + (size_t)h * dk * dv);
    return ORC_OK;
}

int orc_quantize_cols(int64_t n, int dk, int dv, const double *S, int8_t *Z,
                      float *c, float *b)
{
    if (n < 0 || dk <= 0 || dv <= 0 || dv > 1024) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < n; ++h)
        quant_cols(dk, dv, S + (size_t)h * dk * dv, Z + (size_t)h * dk * dv,
                   c + (size_t)h * dk, b + (size_t)h * dv);
    return ORC_OK;
}

int orc_dequantize_cols(int64_t n, int dk, int dv, const int8_t *Z,
                        const float *c, const float *b, double *S)
{
    if (n < 0 || dk <= 0 || dv <= 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < n; ++h)
        dequant_cols(dk, dv, Z + (size_t)h * dk * dv, c + (size_t)h * dk,
                     b + (size_t)h * dv, S + (size_t)h * dk * dv);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Per-window INT8 scheme                                                    */
/* ------------------------------------------------------------------------ */

/*
 * Per-state arrays of the per-window scheme ([LQ] §3.2):
 *   Z    [dk*dv] int8   quantized boundary state (payload of S-hat_0)
 *   s    [dk]    float  its row factors: per-key-row scales (mode 0) or the
 *                       smoothing vector c (mode 1, [LQ] §3.4)
 *   fc   [dv]    float  mode 1: per-value-column scales b (unused in mode 0)
 *   Sw   [dk*dv] double the exact state S_i reached from dequant(S-hat_0)
 *                       by the window's records so far (eq. 3)
 *   rl   [W*dl]  double buffered log-decays  (alpha_i = exp(rl_i))
 *   rk   [W*dk]  double buffered keys        k_i
 *   ru   [W*dv]  double buffered corrections u_i
 *   cnt          number of buffered records, 0 <= cnt < W
 *
 * One token, [LQ] §3.2 eq. 3-4:
 *     u_i = beta (v_i - S_{i-1}^T (alpha_i . k_i))
 *     S_i = Diag(alpha_i) S_{i-1} + k_i u_i^T
 *     y_i = S_i^T q_i                       (read before any quantization)
 *     buffer (alpha_i, k_i, u_i)
 *     at the W-th record: S-hat <- quant_8(S_W), S_W <- dequant(S-hat),
 *     empty the buffer (quant_8 / dequant of the pool's format, `mode`;
 *     with nc compensator pairs, the boundary of §3.3, see boundary()).
 *   ck   [nc*dk], cu [nc*dv] double: the window's compensator pairs.
 */
static void window_one(int mode, int nc, int rec, int dk, int dv, int dl, int W,
                       int8_t *Z, float *s, float *fc, double *ck, double *cu,
                       double *Sw, double *rl, double *rk, double *ru,
                       int32_t *cntp, const float *q, const float *k,
                       const float *v, const float *lam, float beta,
                       double *y, double *r)
{
    const int c = *cntp;
    double u[1024];
    eager_one(0, dk, dv, dl, Sw, q, k, v, lam, beta, y, r, u);
    for (int t = 0; t < dl; ++t) rl[(size_t)c * dl + t] = (double)lam[t];
    for (int i = 0; i < dk; ++i) rk[(size_t)c * dk + i] = stored_key(rec, k[i]);
    for (int j = 0; j < dv; ++j)
        ru[(size_t)c * dv + j] = rec == REC_FP16 ? fp16_round(u[j]) : u[j];
    /* 16-bit records: from here on the state holds the stored record, as a
     * read of the record does (y above used k and u themselves) */
    if (rec == REC_BF16_K)
        for (int i = 0; i < dk; ++i) {
            const double dlt = rk[(size_t)c * dk + i] - (double)k[i];
            for (int j = 0; j < dv; ++j) Sw[(size_t)i * dv + j] += dlt * u[j];
        }
    else if (rec == REC_FP16)
        for (int i = 0; i < dk; ++i) {
            const double kh = rk[(size_t)c * dk + i], kx = (double)k[i];
            for (int j = 0; j < dv; ++j)
                Sw[(size_t)i * dv + j] += kh * ru[(size_t)c * dv + j] - kx * u[j];
        }
    if (c + 1 == W) {
        boundary(mode, nc, rec, dk, dv, Sw, Z, s, fc, ck, cu, 1);
        *cntp = 0;
    } else {
        *cntp = c + 1;
    }
}

static int window_args_ok(int mode, int r, int dk, int dv, int dl, int W)
{
    return valid_dims(dk, dv, dl) && W >= 1 && dk <= 1024 && dv <= 1024 &&
           (mode == 0 || mode == 1) && r >= 0 && r <= 64;
}

/* fc: the column factors ([n_states][dv]); may be NULL in mode 0.  ck, cu:
 * [n_states][nc][dk], [n_states][nc][dv] (nc compensator pairs); may be NULL
 * when nc = 0. */
int orc_window_step(int64_t n, int mode, int nc, int rec, int dk, int dv, int dl, int W,
                    int8_t *Z, float *s, float *fc, double *ck, double *cu,
                    double *Sw, double *rl, double *rk, double *ru,
                    int32_t *cnt, const int64_t *idx, const float *q,
                    const float *k, const float *v, const float *lam,
                    const float *beta, double *y, int nthreads)
{
    if (n < 0 || !window_args_ok(mode, nc, dk, dv, dl, W) || rec < 0 || rec > REC_FP16)
        return ORC_ERR_ARG;
    if ((mode == 1 && fc == NULL) || (nc > 0 && (ck == NULL || cu == NULL)))
        return ORC_ERR_ARG;
    if (n == 0) return ORC_OK;
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel
    {
        double *r = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!r) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t row = 0; row < n; ++row) {
                const int64_t h = idx[row];
                window_one(mode, nc, rec, dk, dv, dl, W, Z + (size_t)h * dk * dv,
                           s + (size_t)h * dk, mode ? fc + (size_t)h * dv : NULL,
                           nc ? ck + (size_t)h * nc * dk : NULL,
                           nc ? cu + (size_t)h * nc * dv : NULL,
                           Sw + (size_t)h * dk * dv,
                           rl + (size_t)h * W * dl, rk + (size_t)h * W * dk,
                           ru + (size_t)h * W * dv, cnt + h, q + row * dk,
                           k + row * dk, v + row * dv, lam + row * dl,
                           beta[row], y + row * dv, r);
            }
        }
        free(r);
    }
    return err ? ORC_ERR_NOMEM : ORC_OK;
}

/* Close the current window early: quantize S_i, start a new window. */
int orc_window_commit(int64_t n, int mode, int r, int rec, int dk, int dv, int8_t *Z,
                      float *s, float *fc, double *ck, double *cu, double *Sw,
                      int32_t *cnt, const int64_t *idx)
{
    if (n < 0 || !window_args_ok(mode, r, dk, dv, 1, 1) || rec < 0 || rec > REC_FP16 ||
        (mode == 1 && fc == NULL) || (r > 0 && (ck == NULL || cu == NULL)))
        return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < n; ++row) {
        const int64_t h = idx[row];
        if (cnt[h] == 0) continue;
        boundary(mode, r, rec, dk, dv, Sw + (size_t)h * dk * dv, Z + (size_t)h * dk * dv,
                 s + (size_t)h * dk, mode ? fc + (size_t)h * dv : NULL,
                 r ? ck + (size_t)h * r * dk : NULL, r ? cu + (size_t)h * r * dv : NULL, 1);
        cnt[h] = 0;
    }
    return ORC_OK;
}

/* Start a window from a given state: S-hat_0 = quant_8(S). */
/* (A load starts the compensator fit from the all-ones vector.) */
int orc_window_load(int64_t n, int mode, int r, int rec, int dk, int dv, const double *S,
                    int8_t *Z, float *s, float *fc, double *ck, double *cu,
                    double *Sw, int32_t *cnt, const int64_t *idx)
{
    if (n < 0 || !window_args_ok(mode, r, dk, dv, 1, 1) || rec < 0 || rec > REC_FP16 ||
        (mode == 1 && fc == NULL) || (r > 0 && (ck == NULL || cu == NULL)))
        return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < n; ++row) {
        const int64_t h = idx[row];
        double *Sh = Sw + (size_t)h * dk * dv;
        for (size_t e = 0; e < (size_t)dk * dv; ++e) Sh[e] = S[(size_t)row * dk * dv + e];
        boundary(mode, r, rec, dk, dv, Sh, Z + (size_t)h * dk * dv, s + (size_t)h * dk,
                 mode ? fc + (size_t)h * dv : NULL, r ? ck + (size_t)h * r * dk : NULL,
                 r ? cu + (size_t)h * r * dv : NULL, 0);
        cnt[h] = 0;
    }
    return ORC_OK;
}

/*
 * Unrolled window state, [LQ] §3.2 eq. 4, from the boundary state and the
 * buffered records alone:
 *   S_l = Gamma_{1:l} S-hat_0 + sum_{j=1..l} Gamma_{j+1:l} k_j u_j^T,
 *   Gamma_{a:b} = Diag(alpha_b) ... Diag(alpha_a), identity when a > b.
 * The diagonal products are accumulated as sums of log-decays.
 */
int orc_window_unrolled(int64_t n, int mode, int r, int dk, int dv, int dl,
                        int W, const int8_t *Z, const float *s, const float *fc,
                        const double *ck, const double *cu, const double *rl,
                        const double *rk, const double *ru, const int32_t *cnt,
                        const int64_t *idx, double *S_out)
{
    if (n < 0 || !window_args_ok(mode, r, dk, dv, dl, W)) return ORC_ERR_ARG;
    if ((mode == 1 && fc == NULL) || (r > 0 && (ck == NULL || cu == NULL)))
        return ORC_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 2)
    for (int64_t row = 0; row < n; ++row) {
        const int64_t h = idx[row];
        const int l = cnt[h];
        const double *RL = rl + (size_t)h * W * dl;
        const double *RK = rk + (size_t)h * W * dk;
        const double *RU = ru + (size_t)h * W * dv;
        double *S = S_out + (size_t)row * dk * dv;
        dequant_mode(mode, dk, dv, Z + (size_t)h * dk * dv, s + (size_t)h * dk,
                     mode ? fc + (size_t)h * dv : NULL, S);
        /* [LQ] eq. 7: the compensator pairs join the boundary state */
        for (int c = 0; c < r; ++c)
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] += ck[((size_t)h * r + c) * dk + i] *
                                             cu[((size_t)h * r + c) * dv + j];
        for (int i = 0; i < dk; ++i) {
            double g = 0.0; /* log of Gamma_{1:l}, row i */
            for (int t = 0; t < l; ++t) g += dlam_at(RL + (size_t)t * dl, dl, i);
            const double G = exp(g);
            for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= G;
        }
        for (int jj = 0; jj < l; ++jj) {
            for (int i = 0; i < dk; ++i) {
                double g = 0.0; /* log of Gamma_{jj+2:l} (records after jj) */
                for (int t = jj + 1; t < l; ++t)
                    g += dlam_at(RL + (size_t)t * dl, dl, i);
                const double a = exp(g) * RK[(size_t)jj * dk + i];
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] += a * RU[(size_t)jj * dv + j];
            }
        }
    }
    return ORC_OK;
}

/*
 * Window readout without forming the state, [LQ] App. B.2 eq. 9 (mode 1:
 * App. B.3 eq. 10, the boundary term B Z^T C Gamma x / 127):
 *   S_l^T x = S-hat_0^T Gamma_{1:l} x + sum_j u_j (k_j^T Gamma_{j+1:l} x).
 * x is [n][dk]; out is [n][dv].
 */
int orc_window_readout(int64_t n, int mode, int r, int dk, int dv, int dl,
                       int W, const int8_t *Z, const float *s, const float *fc,
                       const double *ck, const double *cu, const double *rl,
                       const double *rk, const double *ru, const int32_t *cnt,
                       const int64_t *idx, const double *x, double *out)
{
    if (n < 0 || !window_args_ok(mode, r, dk, dv, dl, W)) return ORC_ERR_ARG;
    if ((mode == 1 && fc == NULL) || (r > 0 && (ck == NULL || cu == NULL)))
        return ORC_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 2)
    for (int64_t row = 0; row < n; ++row) {
        const int64_t h = idx[row];
        const int l = cnt[h];
        const double *RL = rl + (size_t)h * W * dl;
        const double *RK = rk + (size_t)h * W * dk;
        const double *RU = ru + (size_t)h * W * dv;
        const int8_t *Zh = Z + (size_t)h * dk * dv;
        const float *sh = s + (size_t)h * dk;
        const float *bh = mode ? fc + (size_t)h * dv : NULL;
        const double *xr = x + (size_t)row * dk;
        double *o = out + (size_t)row * dv;
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        double ckx[64];
        for (int c = 0; c < r; ++c) ckx[c] = 0.0;
        for (int i = 0; i < dk; ++i) {
            double g = 0.0;
            for (int t = 0; t < l; ++t) g += dlam_at(RL + (size_t)t * dl, dl, i);
            const double gx = exp(g) * xr[i];
            /* [LQ] App. B.3 eq. 10: B Z^T C Gamma x for mode 1 */
            for (int j = 0; j < dv; ++j)
                o[j] += (double)sh[i] * (double)Zh[(size_t)i * dv + j] * gx *
                        (bh ? (double)bh[j] : 1.0);
            for (int c = 0; c < r; ++c) ckx[c] += ck[((size_t)h * r + c) * dk + i] * gx;
        }
        /* eq. 10: + U~ (K~^T Gamma_{1:l} x) */
        for (int c = 0; c < r; ++c)
            for (int j = 0; j < dv; ++j) o[j] += cu[((size_t)h * r + c) * dv + j] * ckx[c];
        for (int jj = 0; jj < l; ++jj) {
            double c = 0.0;
            for (int i = 0; i < dk; ++i) {
                double g = 0.0;
                for (int t = jj + 1; t < l; ++t)
                    g += dlam_at(RL + (size_t)t * dl, dl, i);
                c += RK[(size_t)jj * dk + i] * exp(g) * xr[i];
            }
            for (int j = 0; j < dv; ++j) o[j] += RU[(size_t)jj * dv + j] * c;
        }
    }
    return ORC_OK;
}
