// ls_warp.cuh -- warp-per-head building blocks of the deferred and per-window
// INT8 variants (sm_103a).
//
// One warp owns one (slot, head).  Lane l owns value columns 4l..4l+3 and, for
// vectors indexed by key, key rows 4l..4l+3.  The base is row-major (FP32) or
// in 4x4 quads (INT8, see PoolView), so one warp access covers whole key rows:
// the GEMVs S^T x reduce over key rows inside each lane (no cross-lane
// reduction) and a key row's absmax (the INT8 scale) is a warp reduction.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "ls_device.cuh"
#include "ls_internal.cuh"

namespace ls {

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// L2-coherent loads for data this kernel may have written (the log entry of
// the current token, base rows already folded).
__device__ __forceinline__ float4 ldcg4(const float* p) {
    return __ldcg(reinterpret_cast<const float4*>(p));
}

// Exact INT8 <-> FP32 conversions on the FMA and integer pipes.
// Dequantize: a code n (two's complement byte) biased to u = n + 128 in
// [1, 255] is the low mantissa byte of the FP32 number 2^23 + u; subtracting
// 2^23 + 128 leaves n exactly.
// Quantize: a product t = fl(x f) with |t| < 2^22, plus 1.5 * 2^23, rounds to
// rint(t) (half to even) and leaves it in the low mantissa bits in two's
// complement, so the low byte is the code.  With f = fl(127 / B) and |x| <= B
// (B the row's absmax) |t| < 127.5, so no clamp is needed.
constexpr float kCodeBias = 8388736.0f;     // 2^23 + 128
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

// Byte r of two biased code words (word ^ 0x80808080) as exact FP32 codes.
__device__ __forceinline__ float2 code_values(uint32_t wa, uint32_t wb, int r) {
    const uint32_t sel = 0x7650u | static_cast<uint32_t>(r);
    const float2 b = make_float2(__uint_as_float(__byte_perm(wa, 0x4B000000u, sel)),
                                 __uint_as_float(__byte_perm(wb, 0x4B000000u, sel)));
    return __fadd2_rn(b, make_float2(-kCodeBias, -kCodeBias));
}

// Codes of two values sharing the factor f, as FP32 words whose low byte is
// the code.
__device__ __forceinline__ float2 code_words(float2 x, float f) {
    return __fadd2_rn(__fmul2_rn(x, make_float2(f, f)), make_float2(kRoundMagic, kRoundMagic));
}

// Codes of two values with their own factors (value columns of one row).
__device__ __forceinline__ float2 code_words2(float2 x, float2 f) {
    return __fadd2_rn(__fmul2_rn(x, f), make_float2(kRoundMagic, kRoundMagic));
}

// Low bytes of four words packed little-endian into one word.
__device__ __forceinline__ uint32_t pack_low_bytes(float a, float b, float c, float d) {
    return __byte_perm(__byte_perm(__float_as_uint(a), __float_as_uint(b), 0x0040),
                       __byte_perm(__float_as_uint(c), __float_as_uint(d), 0x0040), 0x5410);
}

// INT8 base, column quads: the 16 bytes of quad (i4, c) hold key rows
// 4*i4..4*i4+3 of value columns 4*c..4*c+3; word m is column 4*c + m and its
// byte r is row 4*i4 + r.  quad_slot / quad_index address the quad in 16-byte
// units.
__host__ __device__ __forceinline__ int quad_slot(int i4, int c) { return i4 * (kD / 4) + c; }
__device__ __forceinline__ size_t quad_index(size_t hd, int i4, int c) {
    return hd * (kD * kD / 16) + static_cast<size_t>(quad_slot(i4, c));
}

// Row r of a quad, dequantized with the factor e: (columns 0, 1), (2, 3).
__device__ __forceinline__ void quad_row(uint4 qb, int r, float e, float2& lo, float2& hi) {
    const float2 ee = make_float2(e, e);
    lo = __fmul2_rn(code_values(qb.x, qb.y, r), ee);
    hi = __fmul2_rn(code_values(qb.z, qb.w, r), ee);
}

// The same with per-column factors b01 (columns 0, 1) and b23 (2, 3) too.
__device__ __forceinline__ void quad_row_cols(uint4 qb, int r, float e, float2 b01, float2 b23, float2& lo,
                                              float2& hi) {
    const float2 ee = make_float2(e, e);
    lo = __fmul2_rn(__fmul2_rn(code_values(qb.x, qb.y, r), b01), ee);
    hi = __fmul2_rn(__fmul2_rn(code_values(qb.z, qb.w, r), b23), ee);
}

// Codes of rows r0..r0+3 x 4 columns (row r = (lo[r], hi[r]) = columns
// 0..3, with its own factor f[r - r0]) packed as one column quad (word m =
// column m, byte r - r0 = row r).
template <int N>
__device__ __forceinline__ uint4 pack_quad(const float2 (&lo)[N], const float2 (&hi)[N], int r0,
                                           const float (&f)[4]) {
    float2 a[4], b[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        a[r] = code_words(lo[r0 + r], f[r]);
        b[r] = code_words(hi[r0 + r], f[r]);
    }
    return make_uint4(pack_low_bytes(a[0].x, a[1].x, a[2].x, a[3].x), pack_low_bytes(a[0].y, a[1].y, a[2].y, a[3].y),
                      pack_low_bytes(b[0].x, b[1].x, b[2].x, b[3].x), pack_low_bytes(b[0].y, b[1].y, b[2].y, b[3].y));
}

// Codes of rows r0..r0+3 x 4 columns with one factor per value column (f01 =
// columns 0, 1; f23 = columns 2, 3), packed as one column quad.
template <int N>
__device__ __forceinline__ uint4 pack_quad_cols(const float2 (&lo)[N], const float2 (&hi)[N], int r0,
                                                float2 f01, float2 f23) {
    float2 a[4], b[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        a[r] = code_words2(lo[r0 + r], f01);
        b[r] = code_words2(hi[r0 + r], f23);
    }
    return make_uint4(pack_low_bytes(a[0].x, a[1].x, a[2].x, a[3].x), pack_low_bytes(a[0].y, a[1].y, a[2].y, a[3].y),
                      pack_low_bytes(b[0].x, b[1].x, b[2].x, b[3].x), pack_low_bytes(b[0].y, b[1].y, b[2].y, b[3].y));
}

// Reduction over the 32 lanes of each of 16 per-lane values v[0..15] (one
// per key row), by recursive halving: 16 shuffles instead of 80.  Lane l
// returns the result for row (l >> 1) & 15.  SUM: sum, otherwise max.
template <bool SUM>
__device__ __forceinline__ float warp_reduce16_scatter(float (&v)[16], int lane) {
#pragma unroll
    for (int b = 4, h = 8; b >= 1; --b, h >>= 1) {
        const bool upper = (lane >> b) & 1;
#pragma unroll
        for (int r = 0; r < h; ++r) {
            const float send = upper ? v[r] : v[r + h];
            const float keep = upper ? v[r + h] : v[r];
            const float got = __shfl_xor_sync(0xffffffffu, send, 1 << b);
            v[r] = SUM ? keep + got : fmaxf(keep, got);
        }
    }
    const float got = __shfl_xor_sync(0xffffffffu, v[0], 1);
    return SUM ? v[0] + got : fmaxf(v[0], got);
}
__device__ __forceinline__ float warp_max16_scatter(float (&v)[16], int lane) {
    return warp_reduce16_scatter<false>(v, lane);
}

// Split x (|x| <= 2^30) into 4 signed base-256 digits, x = sum_d d_d 256^d,
// d_d in [-128, 127]; digit d is returned in out[d] (low byte significant).
__device__ __forceinline__ void digits4(int x, int (&out)[4]) {
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        const int lo = ((x + 128) & 0xff) - 128;
        out[d] = lo;
        x = (x - lo) >> 8;
    }
    out[3] = x;
}

// Smoothed per-value-column quantization ("LeapQuant: Efficient Linear
// Attention with Accurate Recurrent State Quantization", §3.4 eq. 7, App.
// B.3) of the 128 x 128 state a CTA holds in the fold layout: warp w has key
// rows 16w..16w+15, lane l value columns 4l..4l+3 (lo = columns 4l, 4l+1,
// hi = 4l+2, 4l+3).  Per key row, c = max(sqrt(mean |S|), 2^-20) (row sums
// by a reduce-scatter), g = 1 / c, R = S g; per value column, the absmax of R
// over all rows (shared memory across warps) gives b = B / 127 and the
// factor f = 127 / B; codes rint(R f).  Writes the codes of state hd, c to
// rowf[128] and b to colf[128].  red: kWarps * kD floats, fcol: kD floats of
// shared memory.  lo / hi are overwritten with R.
constexpr float kSmoothFloor = 9.5367431640625e-07f;  // 2^-20

__device__ __forceinline__ void quantize_cols_cta(float2 (&lo)[16], float2 (&hi)[16], void* base, size_t hd,
                                                  float* rowf, float* colf, float* red, float* fcol) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i0 = 16 * warp;
    float v[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
        v[r] = (fabsf(lo[r].x) + fabsf(lo[r].y)) + (fabsf(hi[r].x) + fabsf(hi[r].y));
    float c = sqrtf(warp_reduce16_scatter<true>(v, lane) * (1.0f / kD));
    if (!(c >= kSmoothFloor)) c = kSmoothFloor;
    const float g = __fdiv_rn(1.0f, c);
    if ((lane & 1) == 0) rowf[i0 + (lane >> 1)] = c;
    float4 cm = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float gr = __shfl_sync(0xffffffffu, g, 2 * r);
        lo[r] = __fmul2_rn(lo[r], make_float2(gr, gr));
        hi[r] = __fmul2_rn(hi[r], make_float2(gr, gr));
        cm = make_float4(fmaxf(cm.x, fabsf(lo[r].x)), fmaxf(cm.y, fabsf(lo[r].y)), fmaxf(cm.z, fabsf(hi[r].x)),
                         fmaxf(cm.w, fabsf(hi[r].y)));
    }
    reinterpret_cast<float4*>(red)[warp * (kD / 4) + lane] = cm;
    __syncthreads();
    if (tid < kD) {
        float B = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) B = fmaxf(B, red[w * kD + tid]);
        float b, f;
        row_quant_params(B, b, f);
        colf[tid] = b;
        fcol[tid] = f;
    }
    __syncthreads();
    const float4 f4 = reinterpret_cast<const float4*>(fcol)[lane];
#pragma unroll
    for (int qd = 0; qd < 4; ++qd)
        reinterpret_cast<uint4*>(base)[quad_index(hd, i0 / 4 + qd, lane)] =
            pack_quad_cols(lo, hi, 4 * qd, make_float2(f4.x, f4.y), make_float2(f4.z, f4.w));
}

// Per-key-row INT8 quantization of the CTA-held state (fold layout): row
// absmax by a warp reduce-scatter, one division pair per row, codes packed
// into column quads; writes the codes of state hd and the scales to scale[128].
__device__ __forceinline__ void quantize_rows_cta(const float2 (&lo)[16], const float2 (&hi)[16], void* base,
                                                  size_t hd, float* scale) {
    const int lane = threadIdx.x & 31, i0 = 16 * (threadIdx.x >> 5);
    float mx[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
        mx[r] = fmaxf(fmaxf(fabsf(lo[r].x), fabsf(lo[r].y)), fmaxf(fabsf(hi[r].x), fabsf(hi[r].y)));
    float s_mine, f_mine;
    row_quant_params(warp_max16_scatter(mx, lane), s_mine, f_mine);
    if ((lane & 1) == 0) scale[i0 + (lane >> 1)] = s_mine;
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
        float f[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) f[r] = __shfl_sync(0xffffffffu, f_mine, 2 * (4 * qd + r));
        reinterpret_cast<uint4*>(base)[quad_index(hd, i0 / 4 + qd, lane)] = pack_quad(lo, hi, 4 * qd, f);
    }
}

// out[i] = sum_j S_ij v_j for the CTA-held state (fold layout), v in shared
// memory; written by the even lane of each row.
__device__ __forceinline__ void cta_state_times(const float2 (&lo)[16], const float2 (&hi)[16], const float* v,
                                                float* out) {
    const int lane = threadIdx.x & 31, i0 = 16 * (threadIdx.x >> 5);
    const float4 v4 = reinterpret_cast<const float4*>(v)[lane];
    float part[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
        part[r] = fmaf(lo[r].x, v4.x, fmaf(lo[r].y, v4.y, fmaf(hi[r].x, v4.z, hi[r].y * v4.w)));
    const float t = warp_reduce16_scatter<true>(part, lane);
    if ((lane & 1) == 0) out[i0 + (lane >> 1)] = t;
}

// Compensator Tokens ("LeapQuant: Efficient Linear Attention with Accurate
// Recurrent State Quantization", §3.3 eq. 5-6) fitted by the CTA to the state
// it holds (fold layout) before quantization.  For h = 0..R-1, on the
// residual left by the previous pairs: v = all-ones / sqrt(128); kCompIters
// steps v <- R^T (R v) / ||R^T (R v)|| (v kept when the norm is 0); k~ = R v,
// u~ = v; R -= k~ u~^T; the pair becomes log entry h of state hd with
// log-decay snapshot 0.  Shared scratch: vs, ws, ks [kD], red
// [kWarps * kD], nz [4].  All threads of the CTA call it.
constexpr int kCompIters = 3;

__device__ __forceinline__ void fit_compensators_cta(float2 (&lo)[16], float2 (&hi)[16], const PoolView& pv,
                                                     size_t hd, float* vs, float* ws, float* ks, float* red,
                                                     float* nz) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i0 = 16 * warp;
    const size_t kb = hd * static_cast<size_t>(pv.cap);
    for (int h = 0; h < pv.R; ++h) {
        if (tid < kD) vs[tid] = 0.08838834764831845f;  // 1 / sqrt(128)
        __syncthreads();
#pragma unroll 1
        for (int it = 0; it < kCompIters; ++it) {
            cta_state_times(lo, hi, vs, ws);  // w = R v
            __syncthreads();
            float4 p = make_float4(0.f, 0.f, 0.f, 0.f);  // z = R^T w, this warp's rows
#pragma unroll
            for (int r4 = 0; r4 < 4; ++r4) {
                const float4 w4 = reinterpret_cast<const float4*>(ws)[i0 / 4 + r4];
                const float wr[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int row = 4 * r4 + r;
                    p.x = fmaf(lo[row].x, wr[r], p.x);
                    p.y = fmaf(lo[row].y, wr[r], p.y);
                    p.z = fmaf(hi[row].x, wr[r], p.z);
                    p.w = fmaf(hi[row].y, wr[r], p.w);
                }
            }
            reinterpret_cast<float4*>(red)[warp * (kD / 4) + lane] = p;
            __syncthreads();
            float z = 0.0f;
            if (tid < kD) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) z += red[w * kD + tid];
                const float s2 = warp_sum(z * z);
                if (lane == 0) nz[warp] = s2;
            }
            __syncthreads();
            if (tid < kD) {
                const float n2 = (nz[0] + nz[1]) + (nz[2] + nz[3]);
                if (n2 > 0.0f) vs[tid] = z / sqrtf(n2);
            }
            __syncthreads();
        }
        cta_state_times(lo, hi, vs, ks);  // k~ = R v
        __syncthreads();
        if (pv.rec16) {
            // FP16 pairs: the stored (rounded) pair is the one the residual
            // loses, so the next pair is fitted to what it leaves
            if (tid < kD) {
                ks[tid] = __half2float(__float2half_rn(ks[tid]));
                vs[tid] = __half2float(__float2half_rn(vs[tid]));
            }
            __syncthreads();
        }
        const float4 v4 = reinterpret_cast<const float4*>(vs)[lane];
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
            const float4 k4 = reinterpret_cast<const float4*>(ks)[i0 / 4 + r4];
            const float kr[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = 4 * r4 + r;
                lo[row] = __ffma2_rn(make_float2(-kr[r], -kr[r]), make_float2(v4.x, v4.y), lo[row]);
                hi[row] = __ffma2_rn(make_float2(-kr[r], -kr[r]), make_float2(v4.z, v4.w), hi[row]);
            }
        }
        if (tid < kD) {
            if (pv.rec16) {
                reinterpret_cast<__half*>(pv.klog)[(kb + h) * kD + tid] = __float2half_rn(ks[tid]);
                reinterpret_cast<__half*>(pv.ulog)[(kb + h) * kD + tid] = __float2half_rn(vs[tid]);
            } else {
                pv.klog[(kb + h) * kD + tid] = ks[tid];
                pv.ulog[(kb + h) * kD + tid] = vs[tid];
            }
            if (pv.dl == kD) pv.lamlog[hd * static_cast<size_t>(pv.lam_stride) + h * kD + tid] = 0.0f;
            else if (tid == 0) pv.lamlog[hd * static_cast<size_t>(pv.lam_stride) + h] = 0.0f;
        }
        __syncthreads();  // vs / ks are the next pair's scratch
    }
}

enum FoldMode : int { kFoldCommit = 0, kFoldRead = 1, kFoldStep = 2 };

// The current token of one (request, head) for kFoldStep: k, q, v, lambda at
// ro = row * 128 (lambda: per-key gate only), beta, and the output row.
struct TokenIn {
    const float* k;
    const float* q;
    const float* v;
    const float* lam;
    float beta;
    float* y;
    size_t ro;
};

// ---------------------------------------------------------------------------
// CTA-cooperative fold of one state (256 threads).
//
// Folds the first n log entries of state hd into its base:
//     S[i][:] = exp(lb_i) dequant(B)[i][:] + sum_{l<n} exp(lb_i - Lam_l,i) K_l,i U_l[:]
// ("DeltaLog: Deferred Materialization of Recurrent States for Linear
// Attention Decoding", §3.2 eq. 7; eq. 6 when the log holds the current
// token, whose snapshot equals lb).  lb is the cumulative log-decay the log
// is folded at: per key row at lbg (per-key gate; GLOBAL memory, read through
// L2 because the caller may just have written it) or lb_scalar.
//   kFoldCommit: deferred -> S is the new FP32 base;  INT8 -> per key row
//     B_i = max_j |S_ij|, s_i = B_i / 127, codes rint(S_ij * (127 / B_i))
//     ("LeapQuant: Efficient Linear Attention with Accurate Recurrent State
//     Quantization", §3.2 eq. 4, App. B.3) -- written in place;
//   kFoldRead: S is written to out ([d_k][d_v]) and the pool is unchanged;
//   kFoldStep: the token that closes the window, in one pass over the state.
//     lb = lbar + lambda (lambda per key row from tok.lam, or already in
//     lb_scalar), so S = Diag(alpha) S_{t-1} with S_{t-1} the logical state
//     of the n = W - 1 stored entries.  Then r = S^T k, y0 = S^T q,
//     u = beta (v - r), y = y0 + (k.q) u (LeapQuant App. A; y from the
//     unquantized state), S += k u^T, and S is committed as in kFoldCommit:
//     the merge of DeltaLog eq. 6 and the window end of LeapQuant eq. 4
//     without writing the current token to the log.
// Work split: warp w owns key rows 16w..16w+15 (so a row's absmax is a warp
// reduction), lane l value columns 4l..4l+3; 64 FP32 accumulators per
// thread.  The base tile is staged by bulk asynchronous copies, the log in
// chunks of kFoldChunk entries with (a, a) pairs a = exp(lb - Lam) K for the
// paired FMAs.  Returns false after a copy timeout (flagged; nothing of this
// call is left in flight).
// ---------------------------------------------------------------------------
constexpr int kFoldChunk = 16;

struct FoldSmem {
    unsigned char* tile;  // tile_bytes(INT8)
    float2* a2;           // [kFoldChunk][kD] (a, a); kFoldStep: then partial sums
    float4* u4;           // [kFoldChunk][kD / 4] U as FP32 (FP32 folds: the staged ru)
    float* es;            // [kD] exp(lb_i) (* s_i for INT8)
    float* lp;            // [kD] lb_i (per-key gate)
    float* kv;            // [kD] k, q, v, u of the token (kFoldStep)
    float* qv;
    float* vv;
    float* uv;
    float* misc;          // [4] partial k.q
    float4* rk;           // raw log chunk K [kFoldChunk][kD], U, Lambda
    float4* ru;           //   (per key row, or kFoldChunk scalars)
    float4* rl;
    uint64_t* bar;        // tile copies
    uint64_t* lbar;       // log chunk copies
};

// Log chunks are staged by bulk copies next to the tile (K, U, Lambda of
// kFoldChunk entries), one chunk ahead: the next chunk, or the next state's
// first, is in flight while the current one is folded.
__host__ __device__ constexpr size_t fold_raw_bytes(bool) { return size_t(3) * kFoldChunk * kD * 4; }

// INT8 converts U into u4 (its records may be binary16); an FP32 fold reads
// the staged U in place.
__host__ __device__ constexpr size_t fold_smem_bytes(bool int8) {
    return tile_bytes(int8) + size_t(kFoldChunk) * kD * (int8 ? 12 : 8) + 6 * kD * 4 + 16 + fold_raw_bytes(int8) +
           16;
}

__device__ __forceinline__ FoldSmem fold_smem(unsigned char* base, bool int8) {
    FoldSmem f;
    unsigned char* p = base;
    f.tile = p;
    p += tile_bytes(int8);
    f.a2 = reinterpret_cast<float2*>(p);
    p += size_t(kFoldChunk) * kD * 8;
    f.u4 = nullptr;
    if (int8) {
        f.u4 = reinterpret_cast<float4*>(p);
        p += size_t(kFoldChunk) * kD * 4;
    }
    float* v = reinterpret_cast<float*>(p);
    f.es = v;
    f.lp = v + kD;
    f.kv = v + 2 * kD;
    f.qv = v + 3 * kD;
    f.vv = v + 4 * kD;
    f.uv = v + 5 * kD;
    f.misc = v + 6 * kD;
    p = reinterpret_cast<unsigned char*>(v + 6 * kD + 4);
    f.rk = reinterpret_cast<float4*>(p);
    f.ru = f.rk + kFoldChunk * (kD / 4);
    f.rl = f.ru + kFoldChunk * (kD / 4);
    if (!int8) f.u4 = f.ru;  // FP32 records: U is used where it was staged
    p += fold_raw_bytes(int8);
    f.bar = reinterpret_cast<uint64_t*>(p);
    f.lbar = f.bar + 1;
    return f;
}

// Copy state of the fold's two staging pipelines across the states a CTA
// folds in turn: the completed phases of the tile and log barriers, and
// whether the next state's tile / first log chunk is already in flight.
struct FoldPipe {
    uint32_t tile_phase = 0;
    uint32_t log_phase = 0;
    bool tile_issued = false;
    bool log_issued = false;
};

// Stage the base tile of state hd into fs.tile (thread 0 only); completes
// one phase of fs.bar.
template <bool INT8>
__device__ __forceinline__ void fold_issue_tile(const PoolView& pv, size_t hd, const FoldSmem& fs) {
    constexpr uint32_t kTile = static_cast<uint32_t>(tile_bytes(INT8));
    constexpr uint32_t kPart = kTile / 4;
    const unsigned char* src = reinterpret_cast<const unsigned char*>(pv.base) + hd * kTile;
    fence_proxy_async();  // the staging area was last used by generic loads and stores
    mbar_arrive_expect_tx(fs.bar, kTile);
#pragma unroll
    for (int i = 0; i < 4; ++i) bulk_g2s(fs.tile + i * kPart, src + i * kPart, kPart, fs.bar);
}

// Stage log entries c0 .. c0 + nl - 1 (nl <= kFoldChunk, c0 a multiple of
// kFoldChunk) of state hd into the raw area (thread 0 only, INT8); completes
// one phase of fs.lbar.  Scalar-gate snapshots are copied in whole 16-byte
// groups; the padded snapshot stride keeps them inside the state's row.
template <bool PER_KEY>
__device__ __forceinline__ void fold_issue_log(const PoolView& pv, size_t hd, int c0, int nl,
                                               const FoldSmem& fs) {
    const size_t eo = (hd * static_cast<size_t>(pv.cap) + c0) * kD;
    const uint32_t part = static_cast<uint32_t>(nl) * kVecBytes;
    const size_t lb0 = hd * static_cast<size_t>(pv.lam_stride);
    const uint32_t lam_bytes = PER_KEY ? part : static_cast<uint32_t>((nl + 3) / 4 * 16);
    const uint32_t kpart = static_cast<uint32_t>(nl) * kD * key_bytes(pv);  // 16-bit keys: half
    const uint32_t upart = static_cast<uint32_t>(nl) * kD * val_bytes(pv);
    fence_proxy_async();
    mbar_arrive_expect_tx(fs.lbar, kpart + upart + lam_bytes);
    bulk_g2s(fs.rk, reinterpret_cast<const unsigned char*>(pv.klog) + eo * key_bytes(pv), kpart, fs.lbar);
    bulk_g2s(fs.ru, reinterpret_cast<const unsigned char*>(pv.ulog) + eo * val_bytes(pv), upart, fs.lbar);
    if constexpr (PER_KEY)
        bulk_g2s(fs.rl, pv.lamlog + lb0 + static_cast<size_t>(c0) * kD, part, fs.lbar);
    else
        bulk_g2s(fs.rl, pv.lamlog + lb0 + c0, lam_bytes, fs.lbar);
}

// pp: the pipelines' state (see FoldPipe).  next_hd >= 0: once this state's
// tile is in registers the tile of next_hd is staged, and (INT8) once its
// last log chunk is staged the first next_n log entries of next_hd, so their
// latency hides behind this fold.
// COMP (INT8 pools with compensator pairs): fit the pairs at a commit.
template <bool INT8, bool PER_KEY, int MODE, bool COMP = false>
__device__ bool fold_cta(const PoolView& pv, size_t hd, int n, const float* lbg, float lb_scalar,
                         float* out, const FoldSmem& fs, FoldPipe& pp, const TokenIn& tok,
                         long long next_hd, int next_n) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        if (!pp.tile_issued) fold_issue_tile<INT8>(pv, hd, fs);
        if (!pp.log_issued && n > 0) fold_issue_log<PER_KEY>(pv, hd, 0, min(kFoldChunk, n), fs);
    }
    pp.tile_issued = false;
    const bool log_in_flight = n > 0;  // this state's first chunk
    pp.log_issued = false;
    // decay (and INT8 scale) of every key row, once per CTA (a scalar-gate
    // FP32 fold needs one value only); the token's vectors for kFoldStep
    const int i0 = 16 * warp;
    constexpr bool kRowFactors = INT8 || PER_KEY;
    if (tid < kD) {
        float lb = lb_scalar;
        if constexpr (PER_KEY) {
            lb = __ldcg(lbg + tid);
            if constexpr (MODE == kFoldStep) lb += __ldg(tok.lam + tok.ro + tid);
            fs.lp[tid] = lb;
        }
        if constexpr (kRowFactors) {
            float ee = expf(lb);
            if constexpr (INT8) ee *= __ldcg(pv.scale + hd * kD + tid);
            fs.es[tid] = ee;
        }
        if constexpr (MODE == kFoldStep) {
            const float ki = __ldg(tok.k + tok.ro + tid), qi = __ldg(tok.q + tok.ro + tid);
            fs.kv[tid] = ki;
            fs.qv[tid] = qi;
            fs.vv[tid] = __ldg(tok.v + tok.ro + tid);
            const float kq = warp_sum(ki * qi);
            if (lane == 0) fs.misc[warp] = kq;
        }
    }
    const bool ok = mbar_wait_bounded(fs.bar, pp.tile_phase);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            flag_status(pv.status, kDevTimeout);
            mbar_wait_bounded(fs.bar, pp.tile_phase);
            if (log_in_flight) mbar_wait_bounded(fs.lbar, pp.log_phase);
        }
        __syncthreads();
        return false;
    }
    pp.tile_phase ^= 1u;
    // decayed, dequantized base rows; acc[r] = columns 4l..4l+3 of row i0 + r
    float e[16];
#pragma unroll
    for (int r4 = 0; r4 < 4; ++r4) {
        float4 v;
        if constexpr (kRowFactors) {
            v = reinterpret_cast<const float4*>(fs.es)[i0 / 4 + r4];
        } else {
            const float g = expf(lb_scalar);
            v = make_float4(g, g, g, g);
        }
        e[4 * r4 + 0] = v.x;
        e[4 * r4 + 1] = v.y;
        e[4 * r4 + 2] = v.z;
        e[4 * r4 + 3] = v.w;
    }
    float2 lo[16], hi[16];
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
        if constexpr (INT8) {
            uint4 q = reinterpret_cast<const uint4*>(fs.tile)[quad_slot(i0 / 4 + qd, lane)];
            q.x ^= 0x80808080u;
            q.y ^= 0x80808080u;
            q.z ^= 0x80808080u;
            q.w ^= 0x80808080u;
            if (pv.colf != nullptr) {
                const float4 b4 = ldcg4(pv.colf + hd * kD + 4 * lane);
                const float2 b01 = make_float2(b4.x, b4.y), b23 = make_float2(b4.z, b4.w);
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    quad_row_cols(q, r, e[4 * qd + r], b01, b23, lo[4 * qd + r], hi[4 * qd + r]);
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) quad_row(q, r, e[4 * qd + r], lo[4 * qd + r], hi[4 * qd + r]);
            }
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = 4 * qd + r;
                const float4 b = reinterpret_cast<const float4*>(fs.tile)[(i0 + row) * (kD / 4) + lane];
                lo[row] = make_float2(e[row] * b.x, e[row] * b.y);
                hi[row] = make_float2(e[row] * b.z, e[row] * b.w);
            }
        }
    }
    if (next_hd >= 0) {
        __syncthreads();  // the tile is in registers
        if (tid == 0) fold_issue_tile<INT8>(pv, static_cast<size_t>(next_hd), fs);
        pp.tile_issued = true;
    }
    // + sum_l exp(lb - Lam_l) K_l U_l^T, kFoldChunk entries at a time
#pragma unroll 1
    for (int c0 = 0; c0 < n; c0 += kFoldChunk) {
        const int nl = min(kFoldChunk, n - c0);
        __syncthreads();  // the previous chunk is consumed
        // raw chunk (bulk copies) -> (a, a) pairs (and, INT8, U as FP32); then
        // the next chunk, or the next state's first one, is staged behind it:
        // INT8 right away, FP32 (whose U is read in place) after the updates
        const bool lok = mbar_wait_bounded(fs.lbar, pp.log_phase);
        if (__syncthreads_or(!lok)) {
            if (tid == 0) {
                flag_status(pv.status, kDevTimeout);
                mbar_wait_bounded(fs.lbar, pp.log_phase);
                if (pp.tile_issued) mbar_wait_bounded(fs.bar, pp.tile_phase);
            }
            __syncthreads();
            pp.tile_issued = false;
            return false;
        }
        pp.log_phase ^= 1u;
        // (entry, key-row pair) items: each lane stores one float4 of
        // (a, a) pairs, consecutive lanes consecutive addresses
        for (int idx = tid; idx < nl * (kD / 2); idx += kThreads) {
            const int l = idx >> 6, p = idx & 63;
            float2 K2;
            if (pv.k16) {
                const uint32_t w = reinterpret_cast<const uint32_t*>(fs.rk)[idx];
                K2 = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
            } else if (INT8 && pv.rec16) {
                K2 = __half22float2(reinterpret_cast<const __half2*>(fs.rk)[idx]);
            } else {
                K2 = reinterpret_cast<const float2*>(fs.rk)[idx];
            }
            float2 g;
            if constexpr (PER_KEY) {
                const float2 lm = reinterpret_cast<const float2*>(fs.rl)[idx];
                const float2 lb2 = reinterpret_cast<const float2*>(fs.lp)[p];
                g = make_float2(expf(lb2.x - lm.x), expf(lb2.y - lm.y));
            } else {
                const float gg = expf(lb_scalar - reinterpret_cast<const float*>(fs.rl)[l]);
                g = make_float2(gg, gg);
            }
            const float a0 = g.x * K2.x, a1 = g.y * K2.y;
            reinterpret_cast<float4*>(fs.a2)[idx] = make_float4(a0, a0, a1, a1);
        }
        if constexpr (INT8) {
            for (int idx = tid; idx < nl * (kD / 4); idx += kThreads)
                fs.u4[idx] = val4_at(fs.ru, static_cast<size_t>(idx) * 4, pv);
        }
        __syncthreads();
        const bool more = c0 + kFoldChunk < n;
        const bool next = !more && next_hd >= 0 && next_n > 0;
        if constexpr (INT8) {
            if (tid == 0) {
                if (more)
                    fold_issue_log<PER_KEY>(pv, hd, c0 + kFoldChunk, min(kFoldChunk, n - c0 - kFoldChunk), fs);
                else if (next)
                    fold_issue_log<PER_KEY>(pv, static_cast<size_t>(next_hd), 0, min(kFoldChunk, next_n), fs);
            }
            pp.log_issued = next;
        }
#pragma unroll 2
        for (int l = 0; l < nl; ++l) {
            const float4 u = fs.u4[l * (kD / 4) + lane];
            const float2 u01 = make_float2(u.x, u.y), u23 = make_float2(u.z, u.w);
            const float4* ap = reinterpret_cast<const float4*>(fs.a2 + l * kD + i0);
#pragma unroll
            for (int r2 = 0; r2 < 8; ++r2) {
                const float4 aa = ap[r2];  // (a, a) of rows i0 + 2 r2, i0 + 2 r2 + 1
                const float2 a0 = make_float2(aa.x, aa.y), a1 = make_float2(aa.z, aa.w);
                lo[2 * r2] = __ffma2_rn(a0, u01, lo[2 * r2]);
                hi[2 * r2] = __ffma2_rn(a0, u23, hi[2 * r2]);
                lo[2 * r2 + 1] = __ffma2_rn(a1, u01, lo[2 * r2 + 1]);
                hi[2 * r2 + 1] = __ffma2_rn(a1, u23, hi[2 * r2 + 1]);
            }
        }
        if constexpr (!INT8) {
            __syncthreads();  // the staged U is consumed
            if (tid == 0) {
                if (more)
                    fold_issue_log<PER_KEY>(pv, hd, c0 + kFoldChunk, min(kFoldChunk, n - c0 - kFoldChunk), fs);
                else if (next)
                    fold_issue_log<PER_KEY>(pv, static_cast<size_t>(next_hd), 0, min(kFoldChunk, next_n), fs);
            }
            pp.log_issued = next;
        }
    }
    if constexpr (MODE == kFoldStep) {
        // r = S^T k and y0 = S^T q: per-thread partials over its 16 rows,
        // summed over the 8 warps in shared memory (the staged chunks are
        // consumed; their area holds the partials)
        __syncthreads();
        float2 pk01 = make_float2(0.f, 0.f), pk23 = pk01, pq01 = pk01, pq23 = pk01;
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
            const float4 k4 = reinterpret_cast<const float4*>(fs.kv)[i0 / 4 + r4];
            const float4 q4 = reinterpret_cast<const float4*>(fs.qv)[i0 / 4 + r4];
            const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = 4 * r4 + r;
                const float2 k2 = make_float2(kk[r], kk[r]), q2 = make_float2(qq[r], qq[r]);
                pk01 = __ffma2_rn(lo[row], k2, pk01);
                pk23 = __ffma2_rn(hi[row], k2, pk23);
                pq01 = __ffma2_rn(lo[row], q2, pq01);
                pq23 = __ffma2_rn(hi[row], q2, pq23);
            }
        }
        float4* red = reinterpret_cast<float4*>(fs.a2);  // [2][8 warps][128 columns]
        red[warp * 32 + lane] = make_float4(pk01.x, pk01.y, pk23.x, pk23.y);
        red[(kWarps + warp) * 32 + lane] = make_float4(pq01.x, pq01.y, pq23.x, pq23.y);
        __syncthreads();
        if (tid < kD) {
            const float* rf = reinterpret_cast<const float*>(fs.a2);
            float r = 0.0f, y0 = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                r += rf[w * kD + tid];
                y0 += rf[(kWarps + w) * kD + tid];
            }
            const float kq = (fs.misc[0] + fs.misc[1]) + (fs.misc[2] + fs.misc[3]);
            const float u = pv.plain ? fs.vv[tid] : tok.beta * (fs.vv[tid] - r);
            fs.uv[tid] = u;
            tok.y[tok.ro + tid] = fmaf(kq, u, y0);
        }
        __syncthreads();
        // S += k u^T
        const float4 u = reinterpret_cast<const float4*>(fs.uv)[lane];
        const float2 u01 = make_float2(u.x, u.y), u23 = make_float2(u.z, u.w);
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
            const float4 k4 = reinterpret_cast<const float4*>(fs.kv)[i0 / 4 + r4];
            const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 k2 = make_float2(kk[r], kk[r]);
                lo[4 * r4 + r] = __ffma2_rn(k2, u01, lo[4 * r4 + r]);
                hi[4 * r4 + r] = __ffma2_rn(k2, u23, hi[4 * r4 + r]);
            }
        }
    }
    // write the 16 rows
    if constexpr (MODE == kFoldRead) {
#pragma unroll
        for (int r = 0; r < 16; ++r)
            st4(out + (i0 + r) * kD + 4 * lane, make_float4(lo[r].x, lo[r].y, hi[r].x, hi[r].y));
    } else if constexpr (!INT8) {
#pragma unroll
        for (int r = 0; r < 16; ++r)
            st4(reinterpret_cast<float*>(pv.base) + hd * (kD * kD) + (i0 + r) * kD + 4 * lane,
                make_float4(lo[r].x, lo[r].y, hi[r].x, hi[r].y));
    } else {
        // INT8 window boundary: compensator pairs first, then the residual's
        // codes; the staged chunks are consumed, so their area is scratch
        __syncthreads();
        if constexpr (COMP)
            fit_compensators_cta(lo, hi, pv, hd, fs.kv, fs.qv, fs.vv, reinterpret_cast<float*>(fs.a2), fs.misc);
        if (pv.colf != nullptr)
            quantize_cols_cta(lo, hi, pv.base, hd, pv.scale + hd * kD, pv.colf + hd * kD,
                              reinterpret_cast<float*>(fs.a2), fs.kv);
        else
            quantize_rows_cta(lo, hi, pv.base, hd, pv.scale + hd * kD);
    }
    return true;
}

}  // namespace ls
