// ls_int8_step.cu -- per-window INT8 decode step of libls (sm_103a).
//
// One warp per (request, head), as in the deferred step kernel, but with
// nothing of the window end in it: a token that closes its state's window is
// queued, (state, request row), for window_fold_kernel (ls_mma_fold.cu),
// which runs right after this kernel on the same stream and decodes it there.  CTAs of four warps, four per SM (16 warps, up to 128
// registers per thread, 53 KiB of shared memory per CTA): measured on GB300
// against three CTAs of eight warps with a two-stage ring, two CTAs of eight
// warps, and five or six CTAs of four warps, this shape keeps the most bytes
// in flight per SM and was the fastest for the scalar and the per-key gate.
//
// Per token, with B the INT8 codes, s the key-row scales (or the smoothing
// factors c of the column-scale format, with column scales b), e = exp(lp),
// lp = lbar + lambda ("DeltaLog: Deferred Materialization of Recurrent
// States for Linear Attention Decoding", §3.1 eq. 4):
//   r  = b . B^T (e . s . k) + sum_l U_l (K_l . (exp(lp - Lam_l) . k))
//   y0 = b . B^T (e . s . q) + sum_l U_l (K_l . (exp(lp - Lam_l) . q))
//   u  = beta (v - r),   y = y0 + (k.q) u
//   append (K, U, Lam)[L] = (k, u, lp), lbar = lp, L += 1
// ("LeapQuant: Efficient Linear Attention with Accurate Recurrent State
// Quantization", App. A GDN / KDA rows; §3.2 eq. 3 with the window readout of
// App. B.2 eq. 9 and, for column scales, App. B.3 eq. 10).
//
// The two GEMVs over the codes are integer dot products.  The read vector
// x = e . s . k (and e . s . q) is written in 24-bit fixed point against a
// power of two 2^E above its absmax, x_i = X_i 2^(E - 23), |X_i| < 2^23, and
// X_i as its three two's complement bytes: two unsigned digits and a signed
// top digit.  Each 32-bit code word holds 4 key rows of one value column,
// and dp4a multiplies it by the same 4 rows' digit d (signed x unsigned for
// d < 2) into int32 accumulators, which are exact; sum_d acc_d 256^d is
// formed with one exact integer step and one FMA.  The power-of-two scale
// makes x -> X exact but for the rounding to an integer, at most 2^-23 of
// the absmax per element (2^-22 where X is clamped to 2^23 - 1): the
// precision FP32 itself gives the largest elements, so the GEMV is as
// accurate as an FP32 dequantize-and-FMA loop.
//
// Data movement: every warp streams its head through a private ring of three
// 4 KiB shared-memory stages filled by 1-D bulk copies (cp.async.bulk), one
// mbarrier per stage.  Items, in order:
//   0       k, q, key-row factors (+ lambda and lbar for the per-key gate)
//   1 .. 4  codes, 4 KiB = 32 key rows each
//   5       v, k, q (+ lambda and lbar, + the column scales of the
//           column-scale format) again: what the replay, the correction and
//           the append need after the GEMVs, staged anew (k, q, lambda and
//           lbar from L2) so that no register holds them during the GEMVs
//   then    log chunks: K and U of EPC entries (+ their snapshots), or with
//           split replay U and the precomputed coefficients
// Item 0 and the first code chunk are issued before the log length is read
// (as copies, or with windows of up to 16 tokens as L2 prefetches), so the
// dependent load of the state's metadata overlaps their first reads.
#include <cuda_runtime.h>

#include "ls_device.cuh"
#include "ls_internal.cuh"
#include "ls_warp.cuh"

namespace ls {

namespace {

constexpr int kI8Warps = 4;
constexpr int kI8Threads = 32 * kI8Warps;
constexpr int kI8Ring = 3;
constexpr uint32_t kI8Chunk = 4096;
constexpr int kI8Stage = kI8Chunk + 16;  // a scalar-gate log chunk adds 16 B of snapshots
constexpr int kI8CodeItems = 4;          // 16 KiB of codes, 32 key rows per item
constexpr int kI8TailItem = kI8CodeItems + 1;  // v (+ column scales)
constexpr int kI8LogItem0 = kI8TailItem + 1;   // first log chunk
static_assert(kI8Ring <= kI8LogItem0, "the ring's first fill holds no log chunk");
constexpr int kShortWindow = 16;               // see i8_warp_step: the early copies

struct I8Warp {
    unsigned char ring[kI8Ring][kI8Stage];
    uint4 dig[32][2];  // per 4-row group: digit words (k0, k1, k2, q0), (q1, q2, -, -) of
                       //   the read vectors x.k and x.q; byte r of digit word d =
                       //   digit d of key row 4 g + r
    uint64_t bar[kI8Ring];
};
static_assert(sizeof(I8Warp) % 16 == 0, "per-warp shared block must keep 16-byte alignment");

constexpr size_t i8_smem_bytes() { return kI8Warps * sizeof(I8Warp); }
// 228 KiB of shared memory per SM, 1 KiB of it reserved per CTA
static_assert(4 * (i8_smem_bytes() + 1024) <= 228 * 1024, "four CTAs fit one SM");

template <bool PER_KEY, bool SPLIT>
struct I8Plan {
    // log entries per chunk: K, U (+ Lam for the per-key gate), or with split
    // replay U and the two coefficients
    static constexpr int EPC = SPLIT ? kSplitEntries : (PER_KEY ? 2 : 4);
};
static_assert(kSplitEntries * (kVecBytes + 8) <= kI8Stage, "a split log chunk fits a stage");

// d += sum of the four products of signed bytes of a and unsigned bytes of b.
__device__ __forceinline__ int dp4a_su(int a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// ... signed bytes of both.
__device__ __forceinline__ int dp4a_ss(int a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Prefetch `bytes` (a multiple of 16) at p (16-byte aligned) into L2; nothing
// to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Byte transpose of the low three bytes of four words: byte r of w[d] =
// byte d of x[r].  With x[r] the fixed-point value of key row 4 g + r, w[d]
// is digit d of the group.
__device__ __forceinline__ uint3 byte_transpose3(int x0, int x1, int x2, int x3) {
    const uint32_t a = __byte_perm(x0, x1, 0x5140);  // x0.0 x1.0 x0.1 x1.1
    const uint32_t b = __byte_perm(x0, x1, 0x7362);  // x0.2 x1.2 x0.3 x1.3
    const uint32_t c = __byte_perm(x2, x3, 0x5140);
    const uint32_t d = __byte_perm(x2, x3, 0x7362);
    return make_uint3(__byte_perm(a, c, 0x5410), __byte_perm(a, c, 0x7632), __byte_perm(b, d, 0x5410));
}

// Fixed point of a lane's four values of a read vector against the warp's
// absmax: returns the digit words of rows 4 lane .. 4 lane + 3 and sets
// *unit = 2^(E - 23), the value of one integer step.  2^E is the smallest
// power of two above the absmax, clamped to E >= -96 (smaller vectors are
// written with fewer significant bits; 2^(E - 23) stays a normal number).
// |x 2^(23 - E)| < 2^23, and the rounding can reach 2^23 only from below, so
// X is clamped to 2^23 - 1 to fit three bytes.
__device__ __forceinline__ uint3 fixed_point_digits(float x0, float x1, float x2, float x3, float* unit) {
    const float m = warp_absmax_redux(fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))));
    const int E = max(((__float_as_int(m) >> 23) & 0xff) - 126, -96);
    const float f = __int_as_float((150 - E) << 23);  // 2^(23 - E), exact products below
    *unit = __int_as_float((104 + E) << 23);          // 2^(E - 23)
    constexpr int kTop = (1 << 23) - 1;
    return byte_transpose3(min(__float2int_rn(x0 * f), kTop), min(__float2int_rn(x1 * f), kTop),
                           min(__float2int_rn(x2 * f), kTop), min(__float2int_rn(x3 * f), kTop));
}

// Issue item `it` of head hd into stage it % kI8Ring (lane 0 only).  L (the
// live log length) is used by log chunks only.
template <bool PER_KEY, bool SPLIT, int REC>
__device__ __forceinline__ void i8_issue(I8Warp& ws, const StepArgs& a, int row, size_t hd, int L, int it) {
    constexpr int EPC = I8Plan<PER_KEY, SPLIT>::EPC;
    const PoolView& pv = a.pv;
    unsigned char* dst = ws.ring[it % kI8Ring];
    uint64_t* bar = &ws.bar[it % kI8Ring];
    fence_proxy_async();  // the stage's previous contents were read by the generic proxy
    const size_t ro = static_cast<size_t>(row) * kD;
    if (it == 0) {
        mbar_arrive_expect_tx(bar, (PER_KEY ? 5 : 3) * kVecBytes);
        bulk_g2s(dst, a.k + ro, kVecBytes, bar);
        bulk_g2s(dst + kVecBytes, a.q + ro, kVecBytes, bar);
        bulk_g2s(dst + 2 * kVecBytes, pv.scale + hd * kD, kVecBytes, bar);
        if constexpr (PER_KEY) {
            bulk_g2s(dst + 3 * kVecBytes, a.lam + ro, kVecBytes, bar);
            bulk_g2s(dst + 4 * kVecBytes, pv.lbar + hd * kD, kVecBytes, bar);
        }
    } else if (it <= kI8CodeItems) {
        mbar_arrive_expect_tx(bar, kI8Chunk);
        bulk_g2s(dst,
                 reinterpret_cast<const unsigned char*>(pv.base) + hd * (kD * kD) +
                     static_cast<size_t>(it - 1) * kI8Chunk,
                 kI8Chunk, bar);
    } else if (it == kI8TailItem) {
        const bool cols = pv.colf != nullptr;
        mbar_arrive_expect_tx(bar, ((PER_KEY ? 5 : 3) + (cols ? 1 : 0)) * kVecBytes);
        bulk_g2s(dst, a.v + ro, kVecBytes, bar);
        bulk_g2s(dst + kVecBytes, a.k + ro, kVecBytes, bar);
        bulk_g2s(dst + 2 * kVecBytes, a.q + ro, kVecBytes, bar);
        uint32_t off = 3 * kVecBytes;
        if constexpr (PER_KEY) {
            bulk_g2s(dst + off, a.lam + ro, kVecBytes, bar);
            bulk_g2s(dst + off + kVecBytes, pv.lbar + hd * kD, kVecBytes, bar);
            off += 2 * kVecBytes;
        }
        if (cols) bulk_g2s(dst + off, pv.colf + hd * kD, kVecBytes, bar);
    } else if constexpr (SPLIT) {
        // U of n entries, then the coefficients of all EPC entries (48 B; the
        // row stride is a multiple of EPC, so e0 + EPC stays inside the row)
        const int e0 = (it - kI8LogItem0) * EPC;
        const int n = min(EPC, L - e0);
        const size_t eo = (hd * static_cast<size_t>(pv.cap) + e0) * kD;
        const uint32_t upart = static_cast<uint32_t>(n) * kD * rec_val_bytes(REC);
        mbar_arrive_expect_tx(bar, upart + EPC * 8);
        bulk_g2s(dst, reinterpret_cast<const unsigned char*>(pv.ulog) + eo * rec_val_bytes(REC), upart, bar);
        bulk_g2s(dst + EPC * kVecBytes, a.coef + static_cast<size_t>(row) * a.cstride + e0, EPC * 8, bar);
    } else {
        const int e0 = (it - kI8LogItem0) * EPC;
        const int n = min(EPC, L - e0);
        const size_t eo = (hd * static_cast<size_t>(pv.cap) + e0) * kD;
        const uint32_t part = static_cast<uint32_t>(n) * kVecBytes;
        const uint32_t kpart = static_cast<uint32_t>(n) * kD * rec_key_bytes(REC);
        const uint32_t upart = static_cast<uint32_t>(n) * kD * rec_val_bytes(REC);
        const size_t lb0 = hd * static_cast<size_t>(pv.lam_stride);
        mbar_arrive_expect_tx(bar, kpart + upart + (PER_KEY ? part : 16));
        bulk_g2s(dst, reinterpret_cast<const unsigned char*>(pv.klog) + eo * rec_key_bytes(REC), kpart, bar);
        bulk_g2s(dst + EPC * kVecBytes, reinterpret_cast<const unsigned char*>(pv.ulog) + eo * rec_val_bytes(REC),
                 upart, bar);
        if constexpr (PER_KEY)
            bulk_g2s(dst + 2 * EPC * kVecBytes, pv.lamlog + lb0 + static_cast<size_t>(e0) * kD, part, bar);
        else  // 4 snapshots; e0 is a multiple of 4 and the stride is padded to 4
            bulk_g2s(dst + kI8Chunk, pv.lamlog + lb0 + e0, 16, bar);
    }
}

// Wait (bounded) for item `it` of the warp's ring; warp-uniform result.  On
// a timeout the status is flagged and the items still in flight (it ..
// min(NI, it + kI8Ring) - 1) are waited for, so that no copy lands after the
// warp has left.
__device__ __forceinline__ bool i8_wait(I8Warp& ws, const PoolView& pv, int it, int NI) {
    const bool ok = mbar_wait_bounded(&ws.bar[it % kI8Ring], (it / kI8Ring) & 1);
    if (!__any_sync(0xffffffffu, !ok)) return true;
    if ((threadIdx.x & 31) == 0) {
        flag_status(pv.status, kDevTimeout);
        for (int j = it; j < min(NI, it + kI8Ring); ++j) mbar_wait_bounded(&ws.bar[j % kI8Ring], (j / kI8Ring) & 1);
    }
    __syncwarp();
    return false;
}

// The output row of a head given up after a timeout: NaN.
__device__ __forceinline__ int2 i8_abandon(const StepArgs& a, size_t ro) {
    const float nan = __int_as_float(0x7fc00000);
    st4(a.y + ro, make_float4(nan, nan, nan, nan));
    return make_int2(-1, -1);
}

// One warp decodes request row `row` (one head).  Returns (state index,
// row) when the token closes the state's window and is left to the
// window-end kernel, else (-1, -1).
template <bool PER_KEY, bool SPLIT, int REC>
__device__ __forceinline__ int2 i8_warp_step(const StepArgs& a, I8Warp& ws, int row) {
    constexpr int EPC = I8Plan<PER_KEY, SPLIT>::EPC;
    const int2 none = make_int2(-1, -1);
    const PoolView& pv = a.pv;
    const int lane = threadIdx.x & 31;
    const int H = pv.H, W = pv.cap;  // W: log capacity (window + compensator pairs)
    const int b = row / H, h = row - b * H;
    const size_t ro = static_cast<size_t>(row) * kD + 4 * lane;
    const float4 nan4 = make_float4(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000),
                                    __int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
    const int slot = __ldg(a.slot_idx + b);
    if (slot < 0 || slot >= pv.P) {
        if (lane == 0) flag_status(pv.status, kDevSlotRange);
        st4(a.y + ro, nan4);
        return none;
    }
    const size_t hd = static_cast<size_t>(slot) * H + h;
    // The inputs and the first code chunk do not depend on the log length, so
    // they are on their way while it is read.  A token that closes its window
    // needs neither here, and the warp must wait for every copy it issued
    // before it leaves: with windows of up to kShortWindow tokens, where one
    // token in W closes, they are prefetched into L2 (nothing to wait for) and
    // copied once the log length is known; with longer windows they are
    // copied at once.  Measured on GB300, chained tokens of 256 x 48 heads: W
    // = 8 62.2 against 62.9 us with the early copies, W = 16 62.0 against
    // 62.4 us; 128 x 32 per-key-gate heads, W = 32: 34.5 against 34.3 us with
    // the prefetches.
    const int early = W <= kShortWindow ? 0 : 2;  // items copied before the log length is read
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kI8Ring; ++s) mbar_init(&ws.bar[s], 1);
        mbar_fence_init();
        if (early == 2) {
            i8_issue<PER_KEY, SPLIT, REC>(ws, a, row, hd, 0, 0);
            i8_issue<PER_KEY, SPLIT, REC>(ws, a, row, hd, 0, 1);
        } else {
            bulk_prefetch_l2(a.k + static_cast<size_t>(row) * kD, kVecBytes);
            bulk_prefetch_l2(a.q + static_cast<size_t>(row) * kD, kVecBytes);
            bulk_prefetch_l2(pv.scale + hd * kD, kVecBytes);
            if constexpr (PER_KEY) {
                bulk_prefetch_l2(a.lam + static_cast<size_t>(row) * kD, kVecBytes);
                bulk_prefetch_l2(pv.lbar + hd * kD, kVecBytes);
            }
            bulk_prefetch_l2(reinterpret_cast<const unsigned char*>(pv.base) + hd * (kD * kD), kI8Chunk);
        }
    }
    const int L = pv.len[hd];
    const float beta = __ldg(a.beta + row);
    float lp_scalar = 0.0f;
    if constexpr (!PER_KEY) lp_scalar = pv.lbar[hd] + __ldg(a.lam + row);
    const bool bad = L < 0 || L >= W;  // the pool memory of this state was overwritten
    if (bad || L + 1 == W) {
        // a bad state is skipped; a token that closes its window is left whole
        // (its output, the fold of the W - 1 stored records, the
        // requantization) to the window-end kernel, which reads the codes and
        // records once.  Either way the early copies land before the warp leaves.
        if (lane == 0) {
            if (bad) flag_status(pv.status, kDevBadState);
            for (int s = 0; s < early; ++s)
                if (!mbar_wait_bounded(&ws.bar[s], 0)) flag_status(pv.status, kDevTimeout);
        }
        __syncwarp();
        if (bad) {
            st4(a.y + ro, nan4);
            return none;
        }
        return make_int2(static_cast<int>(hd), row);
    }
    if (lane == 0) {
#pragma unroll
        for (int it = 0; it < kI8Ring; ++it)
            if (it >= early) i8_issue<PER_KEY, SPLIT, REC>(ws, a, row, hd, L, it);
    }
    __syncwarp();
    const int NI = kI8LogItem0 + (L + EPC - 1) / EPC;

    // The items are consumed in straight-line code: the first kI8LogItem0
    // items have fixed kinds, stages and phases, so each one's wait and the
    // copy issued behind it compile to their own few instructions; only the
    // log chunks run in a loop.
    float4 k4, q4, v4, lp4;
    float kq = 0.0f, unit_k = 0.0f, unit_q = 0.0f;
    float2 r01 = make_float2(0.f, 0.f), r23 = r01, y01 = r01, y23 = r01;
    int acck[4][3], accq[4][3];  // [value column m][digit d]
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int d = 0; d < 3; ++d) acck[m][d] = accq[m][d] = 0;

    // item 0: read vectors e . s . k and e . s . q as fixed-point digits
    if (!i8_wait(ws, pv, 0, NI)) return i8_abandon(a, ro);
    {
        const float4* st4p = reinterpret_cast<const float4*>(ws.ring[0]);
        const float4 kk = st4p[lane];
        const float4 qq = st4p[32 + lane];
        const float4 s4 = st4p[64 + lane];  // key-row factors
        float4 es;
        if constexpr (PER_KEY) {
            const float4 lam4 = st4p[96 + lane];
            const float4 lb4 = st4p[128 + lane];
            es = make_float4(expf(lb4.x + lam4.x) * s4.x, expf(lb4.y + lam4.y) * s4.y,
                             expf(lb4.z + lam4.z) * s4.z, expf(lb4.w + lam4.w) * s4.w);
        } else {
            const float e = expf(lp_scalar);
            es = make_float4(e * s4.x, e * s4.y, e * s4.z, e * s4.w);
        }
        const uint3 dk = fixed_point_digits(es.x * kk.x, es.y * kk.y, es.z * kk.z, es.w * kk.w, &unit_k);
        const uint3 dq = fixed_point_digits(es.x * qq.x, es.y * qq.y, es.z * qq.z, es.w * qq.w, &unit_q);
        ws.dig[lane][0] = make_uint4(dk.x, dk.y, dk.z, dq.x);
        reinterpret_cast<uint2*>(&ws.dig[lane][1])[0] = make_uint2(dq.y, dq.z);
    }
    __syncwarp();  // the stage is read and the digits are visible to every lane
    if (lane == 0) i8_issue<PER_KEY, SPLIT, REC>(ws, a, row, hd, L, kI8Ring);

    // items 1 .. 4: exact integer GEMVs over 32 key rows each; the lane keeps
    // its 4 value columns
#pragma unroll
    for (int it = 1; it <= kI8CodeItems; ++it) {
        if (!i8_wait(ws, pv, it, NI)) return i8_abandon(a, ro);
        const uint4* cw4 = reinterpret_cast<const uint4*>(ws.ring[it % kI8Ring]);
        const int g0 = (it - 1) * 8;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const uint4 cw = cw4[g * 32 + lane];
            const uint4 d0 = ws.dig[g0 + g][0];  // k0, k1, k2, q0
            const uint2 d1 = reinterpret_cast<const uint2*>(&ws.dig[g0 + g][1])[0];  // q1, q2
            const int col[4] = {static_cast<int>(cw.x), static_cast<int>(cw.y), static_cast<int>(cw.z),
                                static_cast<int>(cw.w)};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                acck[m][0] = dp4a_su(col[m], d0.x, acck[m][0]);
                acck[m][1] = dp4a_su(col[m], d0.y, acck[m][1]);
                acck[m][2] = dp4a_ss(col[m], d0.z, acck[m][2]);
                accq[m][0] = dp4a_su(col[m], d0.w, accq[m][0]);
                accq[m][1] = dp4a_su(col[m], d1.x, accq[m][1]);
                accq[m][2] = dp4a_ss(col[m], d1.y, accq[m][2]);
            }
        }
        __syncwarp();  // every lane is done with the stage
        if (lane == 0 && it + kI8Ring < NI) i8_issue<PER_KEY, SPLIT, REC>(ws, a, row, hd, L, it + kI8Ring);
    }

    // item 5: v, k, q (+ lambda, lbar, column scales); sum_d acc_d 256^d:
    // digits 0 and 1 pair exactly in int32 (|acc_d| <= 128 * 127 * 255),
    // digit 2 joins in one FMA; then the unit and the column scales (eq. 10:
    // applied to the column sums)
    if (!i8_wait(ws, pv, kI8TailItem, NI)) return i8_abandon(a, ro);
    {
        const float4* st4p = reinterpret_cast<const float4*>(ws.ring[kI8TailItem % kI8Ring]);
        v4 = st4p[lane];
        k4 = st4p[32 + lane];
        q4 = st4p[64 + lane];
        if constexpr (PER_KEY) {
            const float4 lam4 = st4p[96 + lane];
            const float4 lb4 = st4p[128 + lane];
            lp4 = make_float4(lb4.x + lam4.x, lb4.y + lam4.y, lb4.z + lam4.z, lb4.w + lam4.w);
        } else {
            lp4 = make_float4(lp_scalar, lp_scalar, lp_scalar, lp_scalar);
        }
        kq = warp_sum(fmaf(k4.x, q4.x, fmaf(k4.y, q4.y, fmaf(k4.z, q4.z, k4.w * q4.w))));
        const float4 colf4 =
            pv.colf != nullptr ? st4p[(PER_KEY ? 160 : 96) + lane] : make_float4(1.f, 1.f, 1.f, 1.f);
        float rk[4], rq[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int k01 = acck[m][0] + (acck[m][1] << 8), q01 = accq[m][0] + (accq[m][1] << 8);
            rk[m] = fmaf(static_cast<float>(acck[m][2]), 65536.0f, static_cast<float>(k01)) * unit_k;
            rq[m] = fmaf(static_cast<float>(accq[m][2]), 65536.0f, static_cast<float>(q01)) * unit_q;
        }
        r01 = make_float2(rk[0] * colf4.x, rk[1] * colf4.y);
        r23 = make_float2(rk[2] * colf4.z, rk[3] * colf4.w);
        y01 = make_float2(rq[0] * colf4.x, rq[1] * colf4.y);
        y23 = make_float2(rq[2] * colf4.z, rq[3] * colf4.w);
    }
    __syncwarp();
    if (lane == 0 && kI8TailItem + kI8Ring < NI)
        i8_issue<PER_KEY, SPLIT, REC>(ws, a, row, hd, L, kI8TailItem + kI8Ring);

    // items 6 ..: the log chunks
#pragma unroll 1
    for (int it = kI8LogItem0; it < NI; ++it) {
        if (!i8_wait(ws, pv, it, NI)) return i8_abandon(a, ro);
        const unsigned char* st = ws.ring[it % kI8Ring];
        const float4* st4p = reinterpret_cast<const float4*>(st);
        const int e0 = (it - kI8LogItem0) * EPC;
        const int n = min(EPC, L - e0);
        if constexpr (SPLIT) {
            // replay with precomputed coefficients (c_k, c_q) per entry
            const float2* cf = reinterpret_cast<const float2*>(st + EPC * kVecBytes);
            // the chunk carries the coefficients of all EPC entries; only the
            // first n (written by this call's prepare kernel) are read
            for (int e = 0; e < n; ++e) {
                const float4 U4 = rec_val4<REC>(st, static_cast<size_t>(e) * kD + 4 * lane);
                const float2 c = cf[e];
                r01 = make_float2(fmaf(c.x, U4.x, r01.x), fmaf(c.x, U4.y, r01.y));
                r23 = make_float2(fmaf(c.x, U4.z, r23.x), fmaf(c.x, U4.w, r23.y));
                y01 = make_float2(fmaf(c.y, U4.x, y01.x), fmaf(c.y, U4.y, y01.y));
                y23 = make_float2(fmaf(c.y, U4.z, y23.x), fmaf(c.y, U4.w, y23.y));
            }
        } else {
            // replay of this chunk's log entries (LeapQuant eq. 9)
            for (int e = 0; e < n; ++e) {
                const float4 K4 = rec_key4<REC>(st, static_cast<size_t>(e) * kD + 4 * lane);
                const float4 U4 = rec_val4<REC>(st + EPC * kVecBytes, static_cast<size_t>(e) * kD + 4 * lane);
                float ck, cq;
                if constexpr (PER_KEY) {
                    const float4 Lm = st4p[(2 * EPC + e) * 32 + lane];
                    const float ax = K4.x * replay_decay(lp4.x - Lm.x), ay = K4.y * replay_decay(lp4.y - Lm.y);
                    const float az = K4.z * replay_decay(lp4.z - Lm.z), aw = K4.w * replay_decay(lp4.w - Lm.w);
                    ck = warp_sum(fmaf(ax, k4.x, fmaf(ay, k4.y, fmaf(az, k4.z, aw * k4.w))));
                    cq = warp_sum(fmaf(ax, q4.x, fmaf(ay, q4.y, fmaf(az, q4.z, aw * q4.w))));
                } else {
                    const float g = expf(lp4.x - reinterpret_cast<const float*>(st + kI8Chunk)[e]);
                    ck = warp_sum(fmaf(K4.x, k4.x, fmaf(K4.y, k4.y, fmaf(K4.z, k4.z, K4.w * k4.w)))) * g;
                    cq = warp_sum(fmaf(K4.x, q4.x, fmaf(K4.y, q4.y, fmaf(K4.z, q4.z, K4.w * q4.w)))) * g;
                }
                r01 = make_float2(fmaf(ck, U4.x, r01.x), fmaf(ck, U4.y, r01.y));
                r23 = make_float2(fmaf(ck, U4.z, r23.x), fmaf(ck, U4.w, r23.y));
                y01 = make_float2(fmaf(cq, U4.x, y01.x), fmaf(cq, U4.y, y01.y));
                y23 = make_float2(fmaf(cq, U4.z, y23.x), fmaf(cq, U4.w, y23.y));
            }
        }
        __syncwarp();  // every lane is done with the stage
        if (lane == 0 && it + kI8Ring < NI) i8_issue<PER_KEY, SPLIT, REC>(ws, a, row, hd, L, it + kI8Ring);
    }

    // ---- delta correction and output -----------------------------------------
    const float4 u4 = make_float4(beta * (v4.x - r01.x), beta * (v4.y - r01.y), beta * (v4.z - r23.x),
                                  beta * (v4.w - r23.y));
    st4(a.y + ro, make_float4(fmaf(kq, u4.x, y01.x), fmaf(kq, u4.y, y01.y), fmaf(kq, u4.z, y23.x),
                              fmaf(kq, u4.w, y23.y)));

    // ---- append entry L ---------------------------------------------------------
    const size_t eo = (hd * static_cast<size_t>(W) + L) * kD;
    if constexpr (REC == kRecBF16K)
        reinterpret_cast<uint2*>(pv.klog)[(eo >> 2) + lane] = float4_to_bf16x4(k4);
    else if constexpr (REC == kRecFP16)
        reinterpret_cast<uint2*>(pv.klog)[(eo >> 2) + lane] = float4_to_half4(k4);
    else
        st4(pv.klog + eo + 4 * lane, k4);
    if constexpr (REC == kRecFP16)
        reinterpret_cast<uint2*>(pv.ulog)[(eo >> 2) + lane] = float4_to_half4(u4);
    else
        st4(pv.ulog + eo + 4 * lane, u4);
    const size_t lb0 = hd * static_cast<size_t>(pv.lam_stride);
    if constexpr (PER_KEY) {
        st4(pv.lamlog + lb0 + static_cast<size_t>(L) * kD + 4 * lane, lp4);
        st4(pv.lbar + hd * kD + 4 * lane, lp4);
    } else if (lane == 0) {
        pv.lamlog[lb0 + L] = lp4.x;
        pv.lbar[hd] = lp4.x;
    }
    if (lane == 0) pv.len[hd] = L + 1;
    return none;
}

// The queue of closing tokens is appended once per CTA (one atomic for the
// CTA's closing heads), not once per head.
template <bool PER_KEY, bool SPLIT, int REC>
__global__ void __launch_bounds__(kI8Threads, 4) int8_step_kernel(const StepArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int2 closing[kI8Warps];
    pdl_enter();
    const int warp = threadIdx.x >> 5;
    const int row = blockIdx.x * kI8Warps + warp;
    int2 e = make_int2(-1, -1);
    if (row < a.batch * a.pv.H) e = i8_warp_step<PER_KEY, SPLIT, REC>(a, reinterpret_cast<I8Warp*>(smem)[warp], row);
    if ((threadIdx.x & 31) == 0) closing[warp] = e;
    __syncthreads();
    if (threadIdx.x == 0) {
        int n = 0;
#pragma unroll
        for (int w = 0; w < kI8Warps; ++w) n += closing[w].x >= 0 ? 1 : 0;
        if (n > 0) {
            int i = atomicAdd(a.pv.foldq, n);
            int2* const q = reinterpret_cast<int2*>(a.pv.foldq + 4);
#pragma unroll
            for (int w = 0; w < kI8Warps; ++w)
                if (closing[w].x >= 0) q[i++] = closing[w];
        }
    }
}

// Shared memory per CTA, and the largest shared-memory carveout so that four
// CTAs fit an SM.
template <typename K>
cudaError_t prepare_kernel(K kernel) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(i8_smem_bytes()));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

template <bool SPLIT, int REC>
cudaError_t prepare_rec() {
    cudaError_t e = prepare_kernel(int8_step_kernel<false, SPLIT, REC>);
    if (e != cudaSuccess) return e;
    return prepare_kernel(int8_step_kernel<true, SPLIT, REC>);
}

template <bool SPLIT, int REC>
cudaError_t launch_rec(const StepArgs& a, bool per_key, dim3 grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kI8Threads);
    cfg.dynamicSmemBytes = i8_smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return per_key ? cudaLaunchKernelEx(&cfg, int8_step_kernel<true, SPLIT, REC>, a)
                   : cudaLaunchKernelEx(&cfg, int8_step_kernel<false, SPLIT, REC>, a);
}

template <bool SPLIT>
cudaError_t launch_format(const StepArgs& a, bool per_key, dim3 grid, cudaStream_t s) {
    if (a.pv.k16) return launch_rec<SPLIT, kRecBF16K>(a, per_key, grid, s);
    if (a.pv.rec16) return launch_rec<SPLIT, kRecFP16>(a, per_key, grid, s);
    return launch_rec<SPLIT, kRecFP32>(a, per_key, grid, s);
}

}  // namespace

cudaError_t prepare_int8_step_kernels() {
    cudaError_t e;
    if ((e = prepare_rec<false, kRecFP32>()) != cudaSuccess) return e;
    if ((e = prepare_rec<false, kRecBF16K>()) != cudaSuccess) return e;
    if ((e = prepare_rec<false, kRecFP16>()) != cudaSuccess) return e;
    if ((e = prepare_rec<true, kRecFP32>()) != cudaSuccess) return e;
    if ((e = prepare_rec<true, kRecBF16K>()) != cudaSuccess) return e;
    return prepare_rec<true, kRecFP16>();
}

cudaError_t launch_int8_step(const StepArgs& a, bool per_key, bool split, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.batch) * a.pv.H;
    const dim3 grid(static_cast<unsigned>((rows + kI8Warps - 1) / kI8Warps));
    const cudaError_t e = split ? launch_format<true>(a, per_key, grid, s) : launch_format<false>(a, per_key, grid, s);
    if (e != cudaSuccess) return e;
    return launch_window_fold(a, per_key, s);
}

}  // namespace ls
