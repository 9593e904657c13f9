/*
 * abi_closed_form.c -- drives libls through include/ls.h alone: no Python,
 * no PyTorch.  The program owns its device memory (cudaMalloc) and uses the
 * legacy default stream.
 *
 * For every variant and both gates, three decode tokens with unit keys give
 * outputs and states in closed form under the delta rule ("LeapQuant:
 * Efficient Linear Attention with Accurate Recurrent State Quantization",
 * App. A; "DeltaLog: Deferred Materialization of Recurrent States for Linear
 * Attention Decoding", §2.1):
 *
 *     u = beta (v - (D S)^T k),   S' = D S + k u^T,   y = S'^T q.
 *
 * Per state, with key rows a and c = a + 64 (mod 128) and S_0 = 0:
 *   token 1: k = e_a, beta = 1, D = I          ->  S_1 = e_a v1^T,
 *            y1 = q1[a] v1;
 *   token 2: k = e_c, beta = 1/2, D = diag(g)  ->  u = v2 / 2 (row c of D S_1
 *            is 0), S_2 = g_a e_a v1^T + e_c (v2/2)^T,
 *            y2 = g_a q2[a] v1 + q2[c] v2 / 2;
 *   token 3: k = e_a, beta = 1, D = I          ->  u = v3 - g_a v1, so row a of
 *            S_3 is v3 (the delta rule overwrites the key's association) and
 *            y3 = q3[a] v3 + q3[c] v2 / 2.
 * g_a = 1/2 for the scalar gate; the per-key gate uses 1/4 on row a and 1/2
 * on every other row.
 *
 * Tokens 1-3 stay inside one window (W = M = 4), so the INT8 pool serves them
 * from its FP32 records and its outputs are as exact as the FP32 variants'.
 * ls_window_commit then folds the window: the FP32 states read back as S_3,
 * the INT8 state within half a key-row scale (max_j |S_3[i][j]| / 254) per
 * element.  Token 1 goes through ls_decode_step, token 2 through
 * ls_decode_step_host, token 3 through ls_decode_step_split_static (log
 * variants) or ls_decode_step (eager).
 *
 * Exit status 0 when every check passes.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ls.h"

enum { D = 128, P = 3, H = 2, B = 2 };

static int failures = 0;

#define CHECK(cond, ...)                      \
    do {                                      \
        if (!(cond)) {                        \
            fprintf(stderr, "FAIL: " __VA_ARGS__); \
            fprintf(stderr, "\n");            \
            ++failures;                       \
        }                                     \
    } while (0)

#define CUDA_OK(call)                                                              \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_),    \
                    __FILE__, __LINE__);                                           \
            exit(2);                                                               \
        }                                                                          \
    } while (0)

/* uniform in [-1, 1) from a 64-bit linear congruential generator */
static uint64_t rng_state = 12345u;
static float urand(void) {
    rng_state = rng_state * 6364136223846793005ull + 1442695040888963407ull;
    return (float)((double)(rng_state >> 11) / 9007199254740992.0 * 2.0 - 1.0);
}

static void fill(float *x, size_t n) {
    for (size_t i = 0; i < n; ++i) x[i] = urand();
}

/* key row a of request b, head h; c = a + 64 */
static int row_a(int b, int h) { return (5 * b + 17 * h + 3) % D; }
static int row_c(int b, int h) { return (row_a(b, h) + 64) % D; }

/* expected y of request b, head h at token t (1..3), from the closed form */
static void expected_y(int t, int per_key, const float *q, const float *v1, const float *v2,
                       const float *v3, int b, int h, float *out) {
    const size_t o = ((size_t)b * H + h) * D;
    const int a = row_a(b, h), c = row_c(b, h);
    const float ga = per_key ? 0.25f : 0.5f;
    for (int j = 0; j < D; ++j) {
        if (t == 1)
            out[j] = q[o + a] * v1[o + j];
        else if (t == 2)
            out[j] = ga * q[o + a] * v1[o + j] + 0.5f * q[o + c] * v2[o + j];
        else
            out[j] = q[o + a] * v3[o + j] + 0.5f * q[o + c] * v2[o + j];
    }
}

static void token_inputs(int t, int per_key, float *k, float *lam, float *beta) {
    memset(k, 0, sizeof(float) * B * H * D);
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const size_t r = (size_t)b * H + h;
            const int a = row_a(b, h), c = row_c(b, h);
            k[r * D + (t == 2 ? c : a)] = 1.0f;
            beta[r] = t == 2 ? 0.5f : 1.0f;
            if (per_key) {
                for (int i = 0; i < D; ++i)
                    lam[r * D + i] = t == 2 ? (i == a ? logf(0.25f) : logf(0.5f)) : 0.0f;
            } else {
                lam[r] = t == 2 ? logf(0.5f) : 0.0f;
            }
        }
}

static float max_abs(const float *x, size_t n) {
    float m = 0.0f;
    for (size_t i = 0; i < n; ++i) m = fmaxf(m, fabsf(x[i]));
    return m;
}

static void run_case(int variant, int gate) {
    const int per_key = gate == LS_GATE_PER_KEY;
    const int log_variant = variant != LS_EAGER_FP32;
    const char *name = variant == LS_EAGER_FP32 ? "eager" : variant == LS_DEFERRED_FP32 ? "deferred" : "int8";
    const size_t nv = (size_t)B * H * D, nl = per_key ? nv : (size_t)B * H;
    ls_pool_desc desc = {P, H, D, D, variant, gate, log_variant ? 4 : 0, 0u};
    size_t bytes = 0;
    CHECK(ls_pool_required_bytes(&desc, &bytes) == LS_OK, "%s: required_bytes", name);
    void *mem = NULL;
    CUDA_OK(cudaMalloc(&mem, bytes));
    ls_pool *pool = NULL;
    CHECK(ls_pool_create(&desc, mem, bytes, NULL, &pool) == LS_OK && pool != NULL, "%s: create", name);
    if (pool == NULL) {
        cudaFree(mem);
        return;
    }

    const int32_t h_slots[B] = {2, 0};
    float *q[3], *v[3], *k = malloc(sizeof(float) * nv), *lam = malloc(sizeof(float) * nv),
          *beta = malloc(sizeof(float) * B * H), *y = malloc(sizeof(float) * nv),
          *ye = malloc(sizeof(float) * D);
    for (int t = 0; t < 3; ++t) {
        q[t] = malloc(sizeof(float) * nv);
        v[t] = malloc(sizeof(float) * nv);
        fill(q[t], nv);
        fill(v[t], nv);
    }
    int32_t *d_slots;
    float *d_q, *d_k, *d_v, *d_lam, *d_beta, *d_y;
    CUDA_OK(cudaMalloc((void **)&d_slots, sizeof(h_slots)));
    CUDA_OK(cudaMalloc((void **)&d_q, sizeof(float) * nv));
    CUDA_OK(cudaMalloc((void **)&d_k, sizeof(float) * nv));
    CUDA_OK(cudaMalloc((void **)&d_v, sizeof(float) * nv));
    CUDA_OK(cudaMalloc((void **)&d_lam, sizeof(float) * nv));
    CUDA_OK(cudaMalloc((void **)&d_beta, sizeof(float) * B * H));
    CUDA_OK(cudaMalloc((void **)&d_y, sizeof(float) * nv));
    CUDA_OK(cudaMemcpy(d_slots, h_slots, sizeof(h_slots), cudaMemcpyHostToDevice));
    size_t staging_bytes = 0;
    CHECK(ls_step_staging_bytes(pool, B, &staging_bytes) == LS_OK, "%s: staging bytes", name);
    void *staging = NULL;
    CUDA_OK(cudaMalloc(&staging, staging_bytes));

    for (int t = 1; t <= 3; ++t) {
        token_inputs(t, per_key, k, lam, beta);
        int rc;
        if (t == 2) {  /* host buffers, copies inside the library */
            rc = ls_decode_step_host(pool, h_slots, B, q[1], k, v[1], lam, beta, y, staging,
                                     staging_bytes, NULL);
            CUDA_OK(cudaDeviceSynchronize());
        } else {
            CUDA_OK(cudaMemcpy(d_q, q[t - 1], sizeof(float) * nv, cudaMemcpyHostToDevice));
            CUDA_OK(cudaMemcpy(d_k, k, sizeof(float) * nv, cudaMemcpyHostToDevice));
            CUDA_OK(cudaMemcpy(d_v, v[t - 1], sizeof(float) * nv, cudaMemcpyHostToDevice));
            CUDA_OK(cudaMemcpy(d_lam, lam, sizeof(float) * nl, cudaMemcpyHostToDevice));
            CUDA_OK(cudaMemcpy(d_beta, beta, sizeof(float) * B * H, cudaMemcpyHostToDevice));
            if (t == 3 && log_variant)
                rc = ls_decode_step_split_static(pool, d_slots, B, d_q, d_k, d_v, d_lam, d_beta, d_y, NULL);
            else
                rc = ls_decode_step(pool, d_slots, B, d_q, d_k, d_v, d_lam, d_beta, d_y, NULL);
            CUDA_OK(cudaMemcpy(y, d_y, sizeof(float) * nv, cudaMemcpyDeviceToHost));
        }
        CHECK(rc == LS_OK, "%s/%d: token %d returned %s", name, gate, t, ls_error_string(rc));
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h) {
                expected_y(t, per_key, q[t - 1], v[0], v[1], v[2], b, h, ye);
                const float *yg = y + ((size_t)b * H + h) * D;
                const float tol = 2e-5f * (max_abs(ye, D) + 1.0f);
                float err = 0.0f;
                for (int j = 0; j < D; ++j) err = fmaxf(err, fabsf(yg[j] - ye[j]));
                CHECK(err <= tol, "%s/%d: token %d request %d head %d: |y - y_exact| = %g", name, gate,
                      t, b, h, err);
            }
    }

    /* close the window, then read S_3 back: row a = v3, row c = v2 / 2, else 0 */
    if (log_variant) {
        const int rc = ls_window_commit(pool, d_slots, B, NULL);
        CHECK(rc == LS_OK, "%s/%d: commit returned %s", name, gate, ls_error_string(rc));
    }
    const size_t ns = (size_t)B * H * D * D;
    float *d_s, *s = malloc(sizeof(float) * ns), *row = malloc(sizeof(float) * D);
    CUDA_OK(cudaMalloc((void **)&d_s, sizeof(float) * ns));
    {
        const int rc = ls_pool_read(pool, d_slots, B, d_s, NULL);
        CHECK(rc == LS_OK, "%s/%d: read returned %s", name, gate, ls_error_string(rc));
    }
    CUDA_OK(cudaMemcpy(s, d_s, sizeof(float) * ns, cudaMemcpyDeviceToHost));
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const size_t o = ((size_t)b * H + h) * D;
            const int a = row_a(b, h), c = row_c(b, h);
            float worst = 0.0f;
            for (int i = 0; i < D; ++i) {
                for (int j = 0; j < D; ++j)
                    row[j] = i == a ? v[2][o + j] : i == c ? 0.5f * v[1][o + j] : 0.0f;
                /* INT8: half a key-row scale, max_j |S[i][j]| / 254 */
                const float tol = variant == LS_WINDOW_INT8 ? max_abs(row, D) / 254.0f * 1.0001f + 1e-7f
                                                          : 2e-5f;
                const float *sg = s + (o + i) * D;
                for (int j = 0; j < D; ++j) {
                    const float e = fabsf(sg[j] - row[j]);
                    if (e > tol) worst = fmaxf(worst, e);
                }
            }
            CHECK(worst == 0.0f, "%s/%d: request %d head %d: state off by %g", name, gate, b, h, worst);
        }

    int32_t status = -1;
    CHECK(ls_pool_status(pool, NULL, &status) == LS_OK && status == 0, "%s/%d: device status %d", name,
          gate, status);

    ls_pool_destroy(pool);
    cudaFree(d_s);
    cudaFree(staging);
    cudaFree(d_slots);
    cudaFree(d_q);
    cudaFree(d_k);
    cudaFree(d_v);
    cudaFree(d_lam);
    cudaFree(d_beta);
    cudaFree(d_y);
    cudaFree(mem);
    for (int t = 0; t < 3; ++t) {
        free(q[t]);
        free(v[t]);
    }
    free(k);
    free(lam);
    free(beta);
    free(y);
    free(ye);
    free(s);
    free(row);
}

int main(void) {
    CHECK(ls_abi_version() == LS_ABI_VERSION, "library ABI %d, header %d", ls_abi_version(), LS_ABI_VERSION);
    /* argument errors are caught on the host, before any launch */
    ls_pool_desc bad = {P, H, 64, D, LS_EAGER_FP32, LS_GATE_SCALAR, 0, 0u};
    size_t bytes = 0;
    CHECK(ls_pool_required_bytes(&bad, &bytes) == LS_ERR_SIZE, "d_k = 64 accepted");
    CHECK(ls_decode_step(NULL, NULL, 1, NULL, NULL, NULL, NULL, NULL, NULL, NULL) == LS_ERR_INVALID,
          "NULL pool accepted");
    const int variants[3] = {LS_EAGER_FP32, LS_DEFERRED_FP32, LS_WINDOW_INT8};
    const int gates[2] = {LS_GATE_SCALAR, LS_GATE_PER_KEY};
    for (int vi = 0; vi < 3; ++vi)
        for (int gi = 0; gi < 2; ++gi) run_case(variants[vi], gates[gi]);
    if (failures == 0) printf("abi_closed_form: ok\n");
    return failures == 0 ? 0 : 1;
}
