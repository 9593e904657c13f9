// ls_step.cu -- base + log decode-step kernel of libls (sm_103a).
//
// Deferred FP32 / per-window INT8: one warp per (request, head), eight heads
// per CTA and no CTA-wide synchronisation until a window closes (see
// ls_warp.cuh for the layout and the CTA-cooperative fold).
//
// Pages: "LeapQuant: Efficient Linear Attention with Accurate Recurrent State
// Quantization" (App. A GDN/KDA expansions; §3.2 eq. 3-4 and App. B.2 eq. 9
// for the window readout) and "DeltaLog: Deferred Materialization of
// Recurrent States for Linear Attention Decoding" (§3.1 Algorithm 1, eq. 4-7;
// §3.3 on value-tile ownership and the single writer of the shared log
// metadata).
#include <cuda_runtime.h>

#include <type_traits>

#include "ls_device.cuh"
#include "ls_internal.cuh"
#include "ls_warp.cuh"

namespace ls {

namespace {

// ---------------------------------------------------------------------------
// (b) deferred FP32 / (c) per-window INT8: base + log step, one warp per head.
//   lp = lbar + lambda (cumulative log-decay after this token, DeltaLog eq. 4)
//   r  = B^T (e . s . k) + sum_l U_l (K_l . (exp(lp - Lam_l) . k))
//   y0 = B^T (e . s . q) + sum_l U_l (K_l . (exp(lp - Lam_l) . q))
//        (B the base, e = exp(lp), s = INT8 key-row scales or 1; the log sum
//         is the window readout of LeapQuant App. B.2 eq. 9 / DeltaLog eq. 7)
//   u  = beta (v - r),   y = y0 + (k.q) u
//   append (K, U, Lam)[L] = (k, u, lp), lbar = lp, L += 1     (DeltaLog eq. 5)
//   on the window's last token the log is folded into the base (DeltaLog
//   eq. 6; LeapQuant eq. 4 + requantization), with y formed from the
//   unquantized state: a deferred pool's CTA decodes that token in one pass
//   over each closing head; an INT8 pool with column scales or compensator
//   pairs appends the token, then the CTA folds the head.  (INT8 pools with
//   per-row scales and no pairs use the kernels of ls_int8_step.cu and
//   ls_mma_fold.cu instead.)
//
// Data movement: every warp streams its head through a private ring of
// kRing shared-memory stages with 1-D bulk asynchronous copies (TMA,
// cp.async.bulk), one mbarrier per stage.  Lane 0 issues, all lanes consume,
// and up to kRing chunks of 4 KiB stay in flight per warp whatever the
// window length.  The items of a head, in order:
//   0          token inputs: k, q, v (+ lambda, lbar for the per-key gate,
//              + key-row scales for INT8)
//   1 .. NT    base chunks of 4 KiB (32 INT8 rows / 8 FP32 rows)
//   then       log chunks: K and U of EPC entries (+ their snapshots)
// The warp is the single writer of its head's log metadata.
//
// Split replay (DeltaLog §5.3): a prepare kernel first writes, per (request,
// head), the two replay coefficients of every live entry,
//   c_k[l] = K_l . (exp(lp - Lam_l) . k),   c_q[l] = K_l . (exp(lp - Lam_l) . q),
// into caller scratch [batch * H][cstride] (float2); the step's log chunks
// then carry U and those coefficients only.  The prepare kernel uses the
// fused replay's lane layout and reductions, so both orders produce the same
// bits.  Here one warp owns all d_v columns of a head, so the fused replay
// computes each dot product once (the pages' split removes dot products
// duplicated across value tiles); what the split changes is where the key
// side of the log is read and reduced.
// ---------------------------------------------------------------------------
constexpr int kRing = 3;
constexpr int kChunk = 4096;
constexpr int kStage = kChunk + 16;  // a scalar-gate log chunk adds 16 B of snapshots

struct WarpSmem {
    unsigned char ring[kRing][kStage];
    union {
        float4 xkq[kD];    // FP32 base: per key row i (xk_i, xk_i, xq_i, xq_i), xk = e.k, xq = e.q
        uint4 dig[32][2];  // INT8 base: per 4-row group, base-256 digits of xk ([0]) and xq ([1]):
                           //   word d = digit d of rows 4g..4g+3 (byte r = row 4g + r)
    };
    uint64_t bar[3];
    uint32_t bar_live;  // bar[] initialised by this warp (lane 0 sets it)
    uint32_t pad;
};
static_assert(sizeof(WarpSmem) % 16 == 0, "per-warp shared block must keep 16-byte alignment");
static_assert(kWarps * sizeof(WarpSmem) >= fold_smem_bytes(false) &&
                  kWarps * sizeof(WarpSmem) >= fold_smem_bytes(true),
              "the window-end fold reuses the rings as staging");

constexpr size_t step_smem_bytes() { return kWarps * sizeof(WarpSmem); }

template <bool INT8, bool PER_KEY, bool SPLIT = false>
struct Plan {
    static constexpr int NT = INT8 ? 4 : 16;  // base chunks
    // log entries per chunk: K, U (+ Lam for the per-key gate) each, or with
    // split replay U and the two coefficients
    static constexpr int EPC = SPLIT ? kSplitEntries : (PER_KEY ? 2 : 4);
    static constexpr int ROWS = INT8 ? 32 : 8;  // key rows per base chunk
};
static_assert(kSplitEntries * (kVecBytes + 8) <= kStage, "a split log chunk fits a stage");

// Issue item `it` of head hd into stage it % kRing (lane 0 only).
template <bool INT8, bool PER_KEY, bool SPLIT, int REC>
__device__ __forceinline__ void issue_item(WarpSmem& ws, const StepArgs& a, int row, size_t hd,
                                           int L, int it) {
    using P = Plan<INT8, PER_KEY, SPLIT>;
    const PoolView& pv = a.pv;
    unsigned char* dst = ws.ring[it % kRing];
    uint64_t* bar = &ws.bar[it % kRing];
    fence_proxy_async();  // the stage's previous contents were read by the generic proxy
    if (it == 0) {
        const size_t ro = static_cast<size_t>(row) * kD;
        const bool cols = INT8 && pv.colf != nullptr;
        uint32_t bytes = 3 * kVecBytes + (PER_KEY ? 2 * kVecBytes : 0) + (INT8 ? kVecBytes : 0) +
                         (cols ? kVecBytes : 0);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(dst, a.k + ro, kVecBytes, bar);
        bulk_g2s(dst + kVecBytes, a.q + ro, kVecBytes, bar);
        bulk_g2s(dst + 2 * kVecBytes, a.v + ro, kVecBytes, bar);
        uint32_t off = 3 * kVecBytes;
        if constexpr (PER_KEY) {
            bulk_g2s(dst + off, a.lam + ro, kVecBytes, bar);
            bulk_g2s(dst + off + kVecBytes, pv.lbar + hd * kD, kVecBytes, bar);
            off += 2 * kVecBytes;
        }
        if constexpr (INT8) {
            bulk_g2s(dst + off, pv.scale + hd * kD, kVecBytes, bar);
            if (cols) bulk_g2s(dst + off + kVecBytes, pv.colf + hd * kD, kVecBytes, bar);
        }
    } else if (it <= P::NT) {
        mbar_arrive_expect_tx(bar, kChunk);
        bulk_g2s(dst, reinterpret_cast<const unsigned char*>(pv.base) + hd * tile_bytes(INT8) +
                          static_cast<size_t>(it - 1) * kChunk,
                 kChunk, bar);
    } else if constexpr (SPLIT) {
        // U of n entries, then the coefficients of all EPC entries (48 B; the
        // row stride is a multiple of EPC, so e0 + EPC stays inside the row)
        const int e0 = (it - 1 - P::NT) * P::EPC;
        const int n = min(P::EPC, L - e0);
        const size_t eo = (hd * static_cast<size_t>(pv.cap) + e0) * kD;
        const uint32_t upart = static_cast<uint32_t>(n) * kD * rec_val_bytes(REC);
        mbar_arrive_expect_tx(bar, upart + P::EPC * 8);
        bulk_g2s(dst, reinterpret_cast<const unsigned char*>(pv.ulog) + eo * rec_val_bytes(REC), upart, bar);
        bulk_g2s(dst + P::EPC * kVecBytes, a.coef + static_cast<size_t>(row) * a.cstride + e0,
                 P::EPC * 8, bar);
    } else {
        const int e0 = (it - 1 - P::NT) * P::EPC;
        const int n = min(P::EPC, L - e0);
        const size_t eo = (hd * static_cast<size_t>(pv.cap) + e0) * kD;
        const uint32_t part = static_cast<uint32_t>(n) * kVecBytes;
        const uint32_t kpart = static_cast<uint32_t>(n) * kD * rec_key_bytes(REC);  // 16-bit keys: half
        const uint32_t upart = static_cast<uint32_t>(n) * kD * rec_val_bytes(REC);
        const size_t lb0 = hd * static_cast<size_t>(pv.lam_stride);
        mbar_arrive_expect_tx(bar, kpart + upart + (PER_KEY ? part : 16));
        bulk_g2s(dst, reinterpret_cast<const unsigned char*>(pv.klog) + eo * rec_key_bytes(REC), kpart, bar);
        bulk_g2s(dst + P::EPC * kVecBytes,
                 reinterpret_cast<const unsigned char*>(pv.ulog) + eo * rec_val_bytes(REC), upart, bar);
        if constexpr (PER_KEY)
            bulk_g2s(dst + 2 * P::EPC * kVecBytes, pv.lamlog + lb0 + static_cast<size_t>(e0) * kD,
                     part, bar);
        else  // 4 snapshots; e0 is a multiple of 4 and the stride is padded to 4
            bulk_g2s(dst + kChunk, pv.lamlog + lb0 + e0, 16, bar);
    }
}

// One warp decodes one (request, head) and returns -1, or the state index hd
// when the token closes the head's window (L + 1 == W) and the CTA has work
// left on it:
//   FP32 base: the warp leaves the token to the CTA, which decodes it in one
//     pass over the state (the fold's kFoldStep); *lp_out = lbar + lambda;
//   INT8 base: the warp decodes and appends it like any other token, and the
//     CTA folds the W entries into the base and requantizes; *lp_out = lbar
//     after the token.  The base and log the CTA re-reads were just streamed
//     by the warp and are mostly still in L2, while the per-warp GEMV keeps
//     the integer arithmetic of every other token.
template <bool INT8, bool PER_KEY, bool SPLIT, int REC>
__device__ __forceinline__ long long warp_step(const StepArgs& a, WarpSmem& ws, int row,
                                               float* lp_out) {
    using P = Plan<INT8, PER_KEY, SPLIT>;
    const int lane = threadIdx.x & 31;
    const PoolView& pv = a.pv;
    const int H = pv.H, W = pv.cap;  // W: log capacity (window + compensator pairs)
    const int b = row / H, h = row - b * H;
    const size_t ro = static_cast<size_t>(row) * kD + 4 * lane;
    const float4 nan4 = make_float4(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000),
                                    __int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
    const int slot = __ldg(a.slot_idx + b);
    if (slot < 0 || slot >= pv.P) {
        if (lane == 0) flag_status(pv.status, kDevSlotRange);
        st4(a.y + ro, nan4);
        return -1;
    }
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const int L = pv.len[hd];
    if (L < 0 || L >= W) {  // the pool memory of this state was overwritten
        if (lane == 0) flag_status(pv.status, kDevBadState);
        st4(a.y + ro, nan4);
        return -1;
    }
    if (!INT8 && L + 1 == W) {
        if constexpr (!PER_KEY) *lp_out = pv.lbar[hd] + __ldg(a.lam + row);
        return static_cast<long long>(hd);
    }
    const int NI = 1 + P::NT + (L + P::EPC - 1) / P::EPC;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kRing; ++s) mbar_init(&ws.bar[s], 1);
        ws.bar_live = 1u;
        mbar_fence_init();
        for (int it = 0; it < min(kRing, NI); ++it) issue_item<INT8, PER_KEY, SPLIT, REC>(ws, a, row, hd, L, it);
    }
    const float beta = __ldg(a.beta + row);
    float lp_scalar = 0.0f;
    if constexpr (!PER_KEY) lp_scalar = pv.lbar[hd] + __ldg(a.lam + row);
    __syncwarp();

    float4 k4, q4, v4, lp4;
    float4 colf4 = make_float4(1.f, 1.f, 1.f, 1.f);  // INT8 column-scale format: b of my columns
    float kq = 0.0f;
    float2 r01 = make_float2(0.f, 0.f), r23 = r01, y01 = r01, y23 = r01;
    // INT8: exact integer GEMVs.  xk (and xq) are written in fixed point
    // against their absmax, x_i ~ X_i * sx 2^-30 with |X_i| <= 2^30, and X_i
    // as four signed base-256 digits; dp4a multiplies 4 key rows of one value
    // column by 4 digits at a time into int32 accumulators (|acc| < 2^21).
    int acck[4][4], accq[4][4];
    float sxk = 0.0f, sxq = 0.0f;
    if constexpr (INT8) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int d = 0; d < 4; ++d) acck[m][d] = accq[m][d] = 0;
    }
#pragma unroll 1
    for (int it = 0; it < NI; ++it) {
        const int stg = it % kRing;
        const bool ok = mbar_wait_bounded(&ws.bar[stg], (it / kRing) & 1);
        if (__any_sync(0xffffffffu, !ok)) {
            // a copy did not land: flag, drain what is still in flight, give up
            if (lane == 0) {
                flag_status(pv.status, kDevTimeout);
                for (int j = it; j < min(NI, it + kRing); ++j)
                    mbar_wait_bounded(&ws.bar[j % kRing], (j / kRing) & 1);
            }
            __syncwarp();
            st4(a.y + ro, nan4);
            return -1;
        }
        const unsigned char* st = ws.ring[stg];
        const float4* st4p = reinterpret_cast<const float4*>(st);
        if (it == 0) {
            k4 = st4p[lane];
            q4 = st4p[32 + lane];
            v4 = st4p[64 + lane];
            int off = 96;
            if constexpr (PER_KEY) {
                const float4 lam4 = st4p[off + lane];
                const float4 lb4 = st4p[off + 32 + lane];
                lp4 = make_float4(lb4.x + lam4.x, lb4.y + lam4.y, lb4.z + lam4.z, lb4.w + lam4.w);
                off += 64;
            } else {
                lp4 = make_float4(lp_scalar, lp_scalar, lp_scalar, lp_scalar);
            }
            float4 es = make_float4(expf(lp4.x), expf(lp4.y), expf(lp4.z), expf(lp4.w));
            if constexpr (INT8) {
                // key-row factors: per-row scales, or the smoothing factors c
                // (LeapQuant App. B.3: C Gamma x is the read vector)
                const float4 s4 = st4p[off + lane];
                es = make_float4(es.x * s4.x, es.y * s4.y, es.z * s4.z, es.w * s4.w);
                if (pv.colf != nullptr) colf4 = st4p[off + 32 + lane];
            }
            const float xk[4] = {es.x * k4.x, es.y * k4.y, es.z * k4.z, es.w * k4.w};
            const float xq[4] = {es.x * q4.x, es.y * q4.y, es.z * q4.z, es.w * q4.w};
            if constexpr (INT8) {
                sxk = warp_max(fmaxf(fmaxf(fabsf(xk[0]), fabsf(xk[1])), fmaxf(fabsf(xk[2]), fabsf(xk[3]))));
                sxq = warp_max(fmaxf(fmaxf(fabsf(xq[0]), fabsf(xq[1])), fmaxf(fabsf(xq[2]), fabsf(xq[3]))));
                const float fk = sxk > 0.0f ? __fdiv_rn(1073741824.0f, sxk) : 0.0f;  // 2^30 / sx
                const float fq = sxq > 0.0f ? __fdiv_rn(1073741824.0f, sxq) : 0.0f;
                uint32_t dk[4] = {0u, 0u, 0u, 0u}, dq[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int r = 0; r < 4; ++r) {  // key row 4*lane + r
                    int a[4], c[4];
                    digits4(min(max(__float2int_rn(xk[r] * fk), -1073741824), 1073741824), a);
                    digits4(min(max(__float2int_rn(xq[r] * fq), -1073741824), 1073741824), c);
#pragma unroll
                    for (int d = 0; d < 4; ++d) {
                        dk[d] |= (static_cast<uint32_t>(a[d]) & 0xffu) << (8 * r);
                        dq[d] |= (static_cast<uint32_t>(c[d]) & 0xffu) << (8 * r);
                    }
                }
                ws.dig[lane][0] = make_uint4(dk[0], dk[1], dk[2], dk[3]);
                ws.dig[lane][1] = make_uint4(dq[0], dq[1], dq[2], dq[3]);
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m) ws.xkq[4 * lane + m] = make_float4(xk[m], xk[m], xq[m], xq[m]);
            }
            kq = warp_sum(fmaf(k4.x, q4.x, fmaf(k4.y, q4.y, fmaf(k4.z, q4.z, k4.w * q4.w))));
            __syncwarp();  // xk / xq visible to every lane before the base chunks
        } else if (it <= P::NT) {
            // base GEMVs over this chunk's key rows; the lane keeps its 4 columns
            const int row0 = (it - 1) * P::ROWS;
            if constexpr (INT8) {
#pragma unroll
                for (int g = 0; g < P::ROWS / 4; ++g) {
                    const uint4 cw = reinterpret_cast<const uint4*>(st)[g * 32 + lane];
                    const uint4 dk = ws.dig[row0 / 4 + g][0];
                    const uint4 dq = ws.dig[row0 / 4 + g][1];
                    const int col[4] = {static_cast<int>(cw.x), static_cast<int>(cw.y),
                                        static_cast<int>(cw.z), static_cast<int>(cw.w)};
                    const int kd[4] = {static_cast<int>(dk.x), static_cast<int>(dk.y),
                                       static_cast<int>(dk.z), static_cast<int>(dk.w)};
                    const int qd[4] = {static_cast<int>(dq.x), static_cast<int>(dq.y),
                                       static_cast<int>(dq.z), static_cast<int>(dq.w)};
#pragma unroll
                    for (int m = 0; m < 4; ++m)
#pragma unroll
                        for (int d = 0; d < 4; ++d) {
                            acck[m][d] = __dp4a(col[m], kd[d], acck[m][d]);
                            accq[m][d] = __dp4a(col[m], qd[d], accq[m][d]);
                        }
                }
                if (it == P::NT) {  // all key rows seen: back to floating point
                    // sum_d acc_d 256^d: digits 1 and 2 combine exactly in int32
                    // (|acc| < 2^21), the rest in FP32 (three roundings)
                    const float ck = sxk * 9.31322574615478515625e-10f;  // sx 2^-30
                    const float cq = sxq * 9.31322574615478515625e-10f;
                    float rk[4], rq[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int tk = acck[m][1] + (acck[m][2] << 8);
                        const int tq = accq[m][1] + (accq[m][2] << 8);
                        rk[m] = fmaf(static_cast<float>(acck[m][3]), 16777216.0f,
                                     fmaf(static_cast<float>(tk), 256.0f,
                                          static_cast<float>(acck[m][0]))) * ck;
                        rq[m] = fmaf(static_cast<float>(accq[m][3]), 16777216.0f,
                                     fmaf(static_cast<float>(tq), 256.0f,
                                          static_cast<float>(accq[m][0]))) * cq;
                    }
                    // column-scale format: B Z^T (C Gamma x) / 127, the column
                    // scales applied after the integer sums (eq. 10)
                    rk[0] *= colf4.x, rk[1] *= colf4.y, rk[2] *= colf4.z, rk[3] *= colf4.w;
                    rq[0] *= colf4.x, rq[1] *= colf4.y, rq[2] *= colf4.z, rq[3] *= colf4.w;
                    r01 = make_float2(rk[0], rk[1]);
                    r23 = make_float2(rk[2], rk[3]);
                    y01 = make_float2(rq[0], rq[1]);
                    y23 = make_float2(rq[2], rq[3]);
                }
            } else {
#pragma unroll
                for (int gr = 0; gr < P::ROWS / 4; ++gr) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float4 v = st4p[(4 * gr + m) * 32 + lane];
                        const float4 x = ws.xkq[row0 + 4 * gr + m];  // (xk, xk, xq, xq)
                        const float2 xk = make_float2(x.x, x.y), xq = make_float2(x.z, x.w);
                        const float2 v01 = make_float2(v.x, v.y), v23 = make_float2(v.z, v.w);
                        r01 = __ffma2_rn(v01, xk, r01);
                        r23 = __ffma2_rn(v23, xk, r23);
                        y01 = __ffma2_rn(v01, xq, y01);
                        y23 = __ffma2_rn(v23, xq, y23);
                    }
                }
            }
        } else if constexpr (SPLIT) {
            // replay with precomputed coefficients (c_k, c_q) per entry
            const int e0 = (it - 1 - P::NT) * P::EPC;
            const int n = min(P::EPC, L - e0);
            const float2* cf = reinterpret_cast<const float2*>(st + P::EPC * kVecBytes);
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
            const int e0 = (it - 1 - P::NT) * P::EPC;
            const int n = min(P::EPC, L - e0);
            for (int e = 0; e < n; ++e) {
                const float4 K4 = rec_key4<REC>(st, static_cast<size_t>(e) * kD + 4 * lane);
                const float4 U4 = rec_val4<REC>(st + P::EPC * kVecBytes, static_cast<size_t>(e) * kD + 4 * lane);
                float ck, cq;
                if constexpr (PER_KEY) {
                    const float4 Lm = st4p[(2 * P::EPC + e) * 32 + lane];
                    const float ax = K4.x * replay_decay(lp4.x - Lm.x), ay = K4.y * replay_decay(lp4.y - Lm.y);
                    const float az = K4.z * replay_decay(lp4.z - Lm.z), aw = K4.w * replay_decay(lp4.w - Lm.w);
                    ck = warp_sum(fmaf(ax, k4.x, fmaf(ay, k4.y, fmaf(az, k4.z, aw * k4.w))));
                    cq = warp_sum(fmaf(ax, q4.x, fmaf(ay, q4.y, fmaf(az, q4.z, aw * q4.w))));
                } else {
                    const float g = expf(lp4.x - reinterpret_cast<const float*>(st + kChunk)[e]);
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
        if (lane == 0 && it + kRing < NI) issue_item<INT8, PER_KEY, SPLIT, REC>(ws, a, row, hd, L, it + kRing);
    }

    // ---- delta correction and output -----------------------------------------
    const float4 u4 = pv.plain ? v4
                               : make_float4(beta * (v4.x - r01.x), beta * (v4.y - r01.y),
                                             beta * (v4.z - r23.x), beta * (v4.w - r23.y));
    st4(a.y + ro, make_float4(fmaf(kq, u4.x, y01.x), fmaf(kq, u4.y, y01.y),
                              fmaf(kq, u4.z, y23.x), fmaf(kq, u4.w, y23.y)));

    // ---- append entry L -------------------------------------------------------
    {
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
        if constexpr (PER_KEY) st4(pv.lamlog + lb0 + static_cast<size_t>(L) * kD + 4 * lane, lp4);
        else if (lane == 0) pv.lamlog[lb0 + L] = lp4.x;
    }
    if constexpr (PER_KEY) st4(pv.lbar + hd * kD + 4 * lane, lp4);
    else if (lane == 0) pv.lbar[hd] = lp4.x;
    if (L + 1 < W) {
        if (lane == 0) pv.len[hd] = L + 1;
        return -1;
    }
    *lp_out = lp4.x;
    return static_cast<long long>(hd);  // INT8 window end: the CTA folds the W entries
}

template <bool INT8, bool PER_KEY, bool COMP, bool SPLIT, int REC>
__global__ void __launch_bounds__(kThreads, 2) log_step_kernel(const StepArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ long long fold_hd[kWarps];
    __shared__ float fold_lb[kWarps];
    pdl_enter();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const PoolView& pv = a.pv;
    const int row = blockIdx.x * kWarps + warp;
    float lp = 0.0f;
    long long hd = -1;
    WarpSmem& ws = reinterpret_cast<WarpSmem*>(smem)[warp];
    if (lane == 0) ws.bar_live = 0u;
    __syncwarp();
    if (row < a.batch * pv.H) hd = warp_step<INT8, PER_KEY, SPLIT, REC>(a, ws, row, &lp);
    if (lane == 0) {
        fold_hd[warp] = hd;
        fold_lb[warp] = lp;
    }
    // ---- window ends: the whole CTA decodes each closing head in turn ----------
    // (the ring memory is free now and becomes the fold's staging area)
    if (!__syncthreads_or(hd >= 0)) return;
    if (lane == 0 && ws.bar_live) {
#pragma unroll
        for (int s = 0; s < kRing; ++s) mbar_inval(&ws.bar[s]);
    }
    __syncthreads();
    const FoldSmem fs = fold_smem(smem, INT8);
    if (threadIdx.x == 0) {
        mbar_init(fs.bar, 1);
        mbar_init(fs.lbar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    FoldPipe pp;
    bool ok = true;
    for (int w = 0; w < kWarps; ++w) {
        const long long h = fold_hd[w];
        if (h < 0) continue;
        const int r = blockIdx.x * kWarps + w;
        const size_t st = static_cast<size_t>(h);
        if (ok) {
            long long next = -1;
            int next_w = w;
            for (int w2 = w + 1; w2 < kWarps && next < 0; ++w2) {
                next = fold_hd[w2];
                next_w = w2;
            }
            if constexpr (!INT8) {
                // the next merging head's token vectors, into L2 one head ahead
                // (k, q, v, and for the per-key gate lambda and lbar: 4 lines each)
                if (next >= 0 && threadIdx.x < (PER_KEY ? 20 : 12)) {
                    const int vec = threadIdx.x >> 2;
                    const float* src = vec == 0 ? a.k : vec == 1 ? a.q : vec == 2 ? a.v : vec == 3 ? a.lam : pv.lbar;
                    const size_t row = vec == 4 ? static_cast<size_t>(next) : static_cast<size_t>(blockIdx.x * kWarps + next_w);
                    prefetch_l2(src + row * kD + 32 * (threadIdx.x & 3));
                }
            }
            const TokenIn tok{a.k, a.q, a.v, a.lam, __ldg(a.beta + r), a.y, static_cast<size_t>(r) * kD};
            const float* lbg = pv.lbar + st * (PER_KEY ? kD : 1);
            if constexpr (INT8)
                ok = fold_cta<INT8, PER_KEY, kFoldCommit, COMP>(pv, st, pv.cap, lbg, fold_lb[w], nullptr, fs, pp,
                                                          tok, next, pv.cap);
            else
                ok = fold_cta<INT8, PER_KEY, kFoldStep>(pv, st, pv.W - 1, lbg, fold_lb[w], nullptr, fs, pp,
                                                        tok, next, pv.W - 1);
            __syncthreads();  // every reader of lbar is done
        }
        if (ok) {
            if (PER_KEY) {
                if (threadIdx.x < kD / 4) st4(pv.lbar + st * kD + 4 * threadIdx.x, make_float4(0.f, 0.f, 0.f, 0.f));
            } else if (threadIdx.x == 0) {
                pv.lbar[st] = 0.0f;
            }
            if (threadIdx.x == 0) pv.len[st] = pv.R;  // the new window's compensator pairs
        } else if (!INT8 && threadIdx.x < kD) {  // after a copy timeout (flagged): no output
            a.y[static_cast<size_t>(r) * kD + threadIdx.x] = __int_as_float(0x7fc00000);
        }
    }
}

// Split replay, first kernel: the replay coefficients of every live log entry
// of each (request, head) into a.coef[row * a.cstride + l] (DeltaLog §5.3).
// One warp per head with the fused step's lane layout (lane l holds keys
// 4l..4l+3) and reductions.  Heads with nothing to replay, heads the step
// will flag, FP32 heads whose merge interval closes on this token (the CTA
// decodes those in one pass over the state) and INT8 heads whose window
// closes on a pool with a window-end queue (the window-end kernel decodes
// those) write nothing.
template <bool INT8, bool PER_KEY>
__global__ void __launch_bounds__(kThreads) replay_prepare_kernel(const StepArgs a) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const PoolView& pv = a.pv;
    if (row >= a.batch * pv.H) return;
    const int H = pv.H;
    const int b = row / H, h = row - b * H;
    const int slot = __ldg(a.slot_idx + b);
    if (slot < 0 || slot >= pv.P) return;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const int L = pv.len[hd];
    if (L <= 0 || L >= pv.cap) return;
    if (!INT8 && L + 1 == pv.W) return;
    if (INT8 && pv.foldq != nullptr && L + 1 == pv.cap) return;
    const size_t ro = static_cast<size_t>(row) * kD + 4 * lane;
    const float4 k4 = __ldg(reinterpret_cast<const float4*>(a.k + ro));
    const float4 q4 = __ldg(reinterpret_cast<const float4*>(a.q + ro));
    float4 lp4;
    if constexpr (PER_KEY) {
        const float4 lam4 = __ldg(reinterpret_cast<const float4*>(a.lam + ro));
        const float4 lb4 = *reinterpret_cast<const float4*>(pv.lbar + hd * kD + 4 * lane);
        lp4 = make_float4(lb4.x + lam4.x, lb4.y + lam4.y, lb4.z + lam4.z, lb4.w + lam4.w);
    } else {
        const float lps = pv.lbar[hd] + __ldg(a.lam + row);
        lp4 = make_float4(lps, lps, lps, lps);
    }
    const size_t lb0 = hd * static_cast<size_t>(pv.lam_stride);
    const size_t e0 = hd * static_cast<size_t>(pv.cap) * kD;
    float2* out = a.coef + static_cast<size_t>(row) * a.cstride;
#pragma unroll 2
    for (int e = 0; e < L; ++e) {
        const size_t eo = e0 + static_cast<size_t>(e) * kD;
        const float4 K4 = key4_at(pv.klog, eo + 4 * lane, pv);
        float ck, cq;
        if constexpr (PER_KEY) {
            const float4 Lm = *reinterpret_cast<const float4*>(pv.lamlog + lb0 + static_cast<size_t>(e) * kD +
                                                                4 * lane);
            const float ax = K4.x * replay_decay(lp4.x - Lm.x), ay = K4.y * replay_decay(lp4.y - Lm.y);
            const float az = K4.z * replay_decay(lp4.z - Lm.z), aw = K4.w * replay_decay(lp4.w - Lm.w);
            ck = warp_sum(fmaf(ax, k4.x, fmaf(ay, k4.y, fmaf(az, k4.z, aw * k4.w))));
            cq = warp_sum(fmaf(ax, q4.x, fmaf(ay, q4.y, fmaf(az, q4.z, aw * q4.w))));
        } else {
            const float g = expf(lp4.x - pv.lamlog[lb0 + e]);
            ck = warp_sum(fmaf(K4.x, k4.x, fmaf(K4.y, k4.y, fmaf(K4.z, k4.z, K4.w * k4.w)))) * g;
            cq = warp_sum(fmaf(K4.x, q4.x, fmaf(K4.y, q4.y, fmaf(K4.z, q4.z, K4.w * q4.w)))) * g;
        }
        if (lane == 0) out[e] = make_float2(ck, cq);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
}

// The record formats a (variant, compensator) pair offers: bfloat16 keys
// without compensator pairs; binary16 records for INT8 only.
template <bool INT8, bool COMP, int REC>
constexpr bool rec_valid() {
    return REC == kRecFP32 || (REC == kRecBF16K && !COMP) || (REC == kRecFP16 && INT8);
}

template <bool INT8, bool COMP, bool SPLIT, int REC>
cudaError_t prepare_rec() {
    if constexpr (rec_valid<INT8, COMP, REC>()) {
        cudaError_t e = set_smem(log_step_kernel<INT8, false, COMP, SPLIT, REC>, step_smem_bytes());
        if (e != cudaSuccess) return e;
        return set_smem(log_step_kernel<INT8, true, COMP, SPLIT, REC>, step_smem_bytes());
    } else {
        return cudaSuccess;
    }
}

template <bool INT8, bool COMP, bool SPLIT>
cudaError_t prepare_formats() {
    cudaError_t e;
    if ((e = prepare_rec<INT8, COMP, SPLIT, kRecFP32>()) != cudaSuccess) return e;
    if ((e = prepare_rec<INT8, COMP, SPLIT, kRecBF16K>()) != cudaSuccess) return e;
    return prepare_rec<INT8, COMP, SPLIT, kRecFP16>();
}

template <bool INT8, bool COMP, bool SPLIT, int REC>
cudaError_t launch_rec(const StepArgs& a, bool per_key, dim3 grid, cudaStream_t s) {
    if constexpr (rec_valid<INT8, COMP, REC>()) {
        const size_t sm = step_smem_bytes();
        return launch_dependent(per_key ? log_step_kernel<INT8, true, COMP, SPLIT, REC>
                                        : log_step_kernel<INT8, false, COMP, SPLIT, REC>,
                                grid, sm, s, a);
    } else {
        return cudaErrorInvalidValue;  // the descriptor checks exclude this format
    }
}

// The step kernel of a pool: its record format picks the instantiation.
template <bool INT8, bool COMP, bool SPLIT>
cudaError_t launch_step_kernel(const StepArgs& a, bool per_key, dim3 grid, cudaStream_t s) {
    if (a.pv.k16) return launch_rec<INT8, COMP, SPLIT, kRecBF16K>(a, per_key, grid, s);
    if (a.pv.rec16) return launch_rec<INT8, COMP, SPLIT, kRecFP16>(a, per_key, grid, s);
    return launch_rec<INT8, COMP, SPLIT, kRecFP32>(a, per_key, grid, s);
}

}  // namespace

cudaError_t prepare_log_step_kernels() {
    cudaError_t e;
    if ((e = prepare_formats<false, false, false>()) != cudaSuccess) return e;
    if ((e = prepare_formats<true, true, false>()) != cudaSuccess) return e;
    if ((e = prepare_formats<false, false, true>()) != cudaSuccess) return e;
    return prepare_formats<true, true, true>();
}

cudaError_t launch_log_step(const StepArgs& a, bool int8, bool per_key, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.batch) * a.pv.H;
    const dim3 grid(static_cast<unsigned>((rows + kWarps - 1) / kWarps));
    if (!int8) return launch_step_kernel<false, false, false>(a, per_key, grid, s);
    // INT8 without compensator pairs: the INT8 step and window-end kernels;
    // with pairs: this kernel, which also fits them at the window end
    if (a.pv.foldq != nullptr) return launch_int8_step(a, per_key, false, s);
    return launch_step_kernel<true, true, false>(a, per_key, grid, s);
}

cudaError_t launch_log_step_split(const StepArgs& a, bool int8, bool per_key, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.batch) * a.pv.H;
    const dim3 grid(static_cast<unsigned>((rows + kWarps - 1) / kWarps));
    cudaError_t e;
    if (int8)
        e = launch_dependent(per_key ? replay_prepare_kernel<true, true> : replay_prepare_kernel<true, false>,
                             grid, 0, s, a);
    else
        e = launch_dependent(per_key ? replay_prepare_kernel<false, true> : replay_prepare_kernel<false, false>,
                             grid, 0, s, a);
    if (e != cudaSuccess) return e;
    if (!int8) return launch_step_kernel<false, false, true>(a, per_key, grid, s);
    if (a.pv.foldq != nullptr) return launch_int8_step(a, per_key, true, s);
    return launch_step_kernel<true, true, true>(a, per_key, grid, s);
}

}  // namespace ls
