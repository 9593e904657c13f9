// ls_step.cu -- decode-step kernels of libls (sm_103a).
//
// Eager FP32: one CTA of 256 threads decodes one (request, head) per token.
// The head's base tile (S^T: 128 value columns x 128 key rows, FP32 64 KiB or INT8
// 16 KiB) is staged in shared memory by four 1-D bulk asynchronous copies
// (TMA, cp.async.bulk) of one quarter (32 columns) each, completing on four
// mbarriers; the warps consume quarter r as soon as it lands.  Each value
// column is reduced over the 128 key rows by a group of 8 lanes (16 rows per
// lane, 3 shuffle levels) -- the two GEMVs r = S^T(alpha.k), y0 = S^T(alpha.q)
// of the delta-rule step.  Value columns are independent, so no CTA waits on
// another.
//
// Deferred FP32 / per-window INT8: one warp per (request, head), eight heads
// per CTA and no CTA-wide synchronisation (see ls_warp.cuh for the layout).
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

constexpr uint32_t kQuarterF32 = 32 * kD * 4;  // 16 KiB
constexpr uint32_t kQuarterI8 = 32 * kD;       // 4 KiB

// A slot index outside [0, P): flag it, fill the output row with NaN.
__device__ __forceinline__ void skip_bad_row(const StepArgs& a, int row) {
    if (threadIdx.x == 0) flag_status(a.pv.status, kDevSlotRange);
    if (threadIdx.x < kD) a.y[static_cast<size_t>(row) * kD + threadIdx.x] = __int_as_float(0x7fc00000);
}

// Issue the four quarter copies of a tile (thread 0 only).
template <bool INT8>
__device__ __forceinline__ void issue_tile(unsigned char* tile, const unsigned char* gtile,
                                           uint64_t* bars) {
    constexpr uint32_t q = INT8 ? kQuarterI8 : kQuarterF32;
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    mbar_fence_init();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        mbar_arrive_expect_tx(&bars[i], q);
        bulk_g2s(tile + i * q, gtile + i * q, q, &bars[i]);
    }
}

// Bounded wait on quarter r, made uniform over the CTA.  On a timeout the
// CTA flags the status word, drains its own copies (bounded) and must return.
__device__ __forceinline__ bool wait_quarter(uint64_t* bars, int r, int32_t* status) {
    const bool ok = mbar_wait_bounded(&bars[r], 0);
    if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) flag_status(status, kDevTimeout);
#pragma unroll
        for (int i = 0; i < 4; ++i) mbar_wait_bounded(&bars[i], 0);
        return false;
    }
    return true;
}

// ---------------------------------------------------------------------------
// (a) eager FP32: read S, r = S^T(alpha.k), u = beta (v - r),
//     S <- Diag(alpha) S + k u^T (written in place), y = S^T(alpha.q) + (k.q) u
//     (= S_t^T q).  LeapQuant App. A with eq. 1.
// ---------------------------------------------------------------------------
template <bool PER_KEY>
__global__ void __launch_bounds__(kThreads, 3) eager_step_kernel(const StepArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* tile = smem;
    float* xk_s = reinterpret_cast<float*>(smem + tile_bytes(false));
    float* xq_s = xk_s + kD;
    float* al_s = xq_s + kD;
    float* k_s = al_s + kD;
    float* v_s = k_s + kD;
    float* y_s = v_s + kD;
    float* misc = y_s + kD;
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(misc) + kMiscBytes);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    const int H = a.pv.H;
    const int b = row / H, h = row - b * H;
    const int slot = __ldg(a.slot_idx + b);
    if (slot < 0 || slot >= a.pv.P) {
        skip_bad_row(a, row);
        return;
    }
    const size_t hd = static_cast<size_t>(slot) * H + h;
    float* gtile = reinterpret_cast<float*>(a.pv.base) + hd * (kD * kD);
    if (tid == 0) issue_tile<false>(tile, reinterpret_cast<const unsigned char*>(gtile), bars);

    const size_t ro = static_cast<size_t>(row) * kD;
    float kq_part = 0.0f;
    if (tid < kD) {
        const float ki = __ldg(a.k + ro + tid), qi = __ldg(a.q + ro + tid);
        const float lam = PER_KEY ? __ldg(a.lam + ro + tid) : __ldg(a.lam + row);
        const float al = expf(lam);
        xk_s[tid] = al * ki;
        xq_s[tid] = al * qi;
        al_s[tid] = al;
        k_s[tid] = ki;
        v_s[tid] = __ldg(a.v + ro + tid);
        kq_part = ki * qi;
    }
    kq_part = warp_sum(kq_part);
    if (lane == 0 && warp < 4) misc[warp] = kq_part;
    const float beta = __ldg(a.beta + row);
    __syncthreads();
    const float kq = (misc[0] + misc[1]) + (misc[2] + misc[3]);

    const int g = lane & 7, c = lane >> 3;
    float xk[16], xq[16];
    gather16<false>(xk_s, g, xk);
    gather16<false>(xq_s, g, xq);

#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
        const int j = round_col(r, warp, c);
        if (!wait_quarter(bars, r, a.pv.status)) return;
        float s[16];
        load_tile16<false>(tile, j, g, s);
        float rr = 0.0f, yy = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            rr = fmaf(s[e], xk[e], rr);
            yy = fmaf(s[e], xq[e], yy);
        }
        rr = group8_sum(rr);
        yy = group8_sum(yy);
        const float u = beta * (v_s[j] - rr);
        if (g == 0) y_s[j] = fmaf(kq, u, yy);
        float* dst = gtile + j * kD;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int i0 = run_row<false>(g, m);
            const float4 al4 = *reinterpret_cast<const float4*>(al_s + i0);
            const float4 k4 = *reinterpret_cast<const float4*>(k_s + i0);
            float4 o;
            o.x = fmaf(k4.x, u, al4.x * s[4 * m + 0]);
            o.y = fmaf(k4.y, u, al4.y * s[4 * m + 1]);
            o.z = fmaf(k4.z, u, al4.z * s[4 * m + 2]);
            o.w = fmaf(k4.w, u, al4.w * s[4 * m + 3]);
            st4(dst + i0, o);
        }
    }
    __syncthreads();
    if (tid < 32) st4(a.y + ro + 4 * tid, *reinterpret_cast<const float4*>(y_s + 4 * tid));
}

// ---------------------------------------------------------------------------
// (b) deferred FP32 / (c) per-window INT8: base + log step, one warp per head.
//   lp = lbar + lambda (cumulative log-decay after this token, DeltaLog eq. 4)
//   r  = B^T (e . s . k) + sum_l U_l (K_l . (exp(lp - Lam_l) . k))
//   y0 = B^T (e . s . q) + sum_l U_l (K_l . (exp(lp - Lam_l) . q))
//        (B the base, e = exp(lp), s = INT8 key-row scales or 1; the log sum
//         is the window readout of LeapQuant App. B.2 eq. 9 / DeltaLog eq. 7)
//   u  = beta (v - r),   y = y0 + (k.q) u
//   append (K, U, Lam)[L] = (k, u, lp), lbar = lp, L += 1     (DeltaLog eq. 5)
//   on the window's last token the W entries are folded into the base right
//   away by the same warp (DeltaLog eq. 6; LeapQuant eq. 4 + requantization),
//   after y was formed from the unquantized state.
// The warp is the single writer of its head's log metadata.
// ---------------------------------------------------------------------------
template <bool INT8>
struct RowWord {
    using T = typename std::conditional<INT8, uint32_t, float4>::type;
    static __device__ __forceinline__ T load(const void* base, size_t hd, int i, int lane) {
        if constexpr (INT8) {
            const uint32_t* p = reinterpret_cast<const uint32_t*>(base) + hd * (kD * kD / 4) +
                                i * (kD / 4) + lane;
            uint32_t w;
            asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(w) : "l"(p));
            return w;
        } else {
            return ld_stream4(reinterpret_cast<const float*>(base) + hd * (kD * kD) + i * kD +
                              4 * lane);
        }
    }
    static __device__ __forceinline__ float4 values(T w) {
        if constexpr (INT8) {
            return codes4(w);
        } else {
            return w;
        }
    }
};

template <bool INT8, bool PER_KEY>
__global__ void __launch_bounds__(kThreads) log_step_kernel(const StepArgs a) {
    __shared__ __align__(16) float2 xkq_s[kWarps][kD];  // (e s k, e s q) per key row
    __shared__ __align__(16) float lp_s[kWarps][kD];    // lp per key row (per-key gate)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const PoolView& pv = a.pv;
    const int H = pv.H, W = pv.W;
    const int row = blockIdx.x * kWarps + warp;
    if (row >= a.batch * H) return;
    const int b = row / H, h = row - b * H;
    const size_t ro = static_cast<size_t>(row) * kD + 4 * lane;
    const float4 nan4 = make_float4(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000),
                                    __int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
    const int slot = __ldg(a.slot_idx + b);
    if (slot < 0 || slot >= pv.P) {
        if (lane == 0) flag_status(pv.status, kDevSlotRange);
        st4(a.y + ro, nan4);
        return;
    }
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const int L = pv.len[hd];
    if (L < 0 || L >= W) {  // the pool memory of this state was overwritten
        if (lane == 0) flag_status(pv.status, kDevBadState);
        st4(a.y + ro, nan4);
        return;
    }

    // ---- token inputs; lane l holds key rows / value columns 4l..4l+3 ------
    const float4 k4 = ldg4(a.k + ro), q4 = ldg4(a.q + ro), v4 = ldg4(a.v + ro);
    float4 lp4;
    if constexpr (PER_KEY) {
        const float4 lam4 = ldg4(a.lam + ro);
        const float4 lb4 = *reinterpret_cast<const float4*>(pv.lbar + hd * kD + 4 * lane);
        lp4 = make_float4(lb4.x + lam4.x, lb4.y + lam4.y, lb4.z + lam4.z, lb4.w + lam4.w);
    } else {
        const float lp = pv.lbar[hd] + __ldg(a.lam + row);
        lp4 = make_float4(lp, lp, lp, lp);
    }
    const float beta = __ldg(a.beta + row);
    float4 es4 = make_float4(expf(lp4.x), expf(lp4.y), expf(lp4.z), expf(lp4.w));
    if constexpr (INT8) {
        const float4 s4 = *reinterpret_cast<const float4*>(pv.scale + hd * kD + 4 * lane);
        es4 = make_float4(es4.x * s4.x, es4.y * s4.y, es4.z * s4.z, es4.w * s4.w);
    }
    {
        float4* xs = reinterpret_cast<float4*>(&xkq_s[warp][4 * lane]);
        xs[0] = make_float4(es4.x * k4.x, es4.x * q4.x, es4.y * k4.y, es4.y * q4.y);
        xs[1] = make_float4(es4.z * k4.z, es4.z * q4.z, es4.w * k4.w, es4.w * q4.w);
        if constexpr (PER_KEY) *reinterpret_cast<float4*>(&lp_s[warp][4 * lane]) = lp4;
    }
    const float kq = warp_sum(fmaf(k4.x, q4.x, fmaf(k4.y, q4.y, fmaf(k4.z, q4.z, k4.w * q4.w))));
    __syncwarp();

    // ---- base GEMVs: stream the key rows, lane keeps its 4 columns ----------
    float2 r01 = make_float2(0.f, 0.f), r23 = r01, y01 = r01, y23 = r01;
    constexpr int RB = INT8 ? 32 : 8;  // rows in flight per lane (128 B words / 512 B rows)
#pragma unroll 1
    for (int i0 = 0; i0 < kD; i0 += RB) {
        typename RowWord<INT8>::T z[RB];
#pragma unroll
        for (int rr = 0; rr < RB; ++rr) z[rr] = RowWord<INT8>::load(pv.base, hd, i0 + rr, lane);
#pragma unroll
        for (int rr = 0; rr < RB; ++rr) {
            const float2 x = xkq_s[warp][i0 + rr];
            const float4 v = RowWord<INT8>::values(z[rr]);
            const float2 v01 = make_float2(v.x, v.y), v23 = make_float2(v.z, v.w);
            const float2 xk = make_float2(x.x, x.x), xq = make_float2(x.y, x.y);
            r01 = __ffma2_rn(v01, xk, r01);
            r23 = __ffma2_rn(v23, xk, r23);
            y01 = __ffma2_rn(v01, xq, y01);
            y23 = __ffma2_rn(v23, xq, y23);
        }
    }
    float4 r4 = make_float4(r01.x, r01.y, r23.x, r23.y);
    float4 y4 = make_float4(y01.x, y01.y, y23.x, y23.y);

    // ---- replay of the live log ----------------------------------------------
    const size_t e0 = hd * static_cast<size_t>(W);
#pragma unroll 2
    for (int l = 0; l < L; ++l) {
        const size_t eo = (e0 + l) * kD + 4 * lane;
        const float4 K4 = ldg4(pv.klog + eo);
        const float4 U4 = ldg4(pv.ulog + eo);
        float ck, cq;
        if constexpr (PER_KEY) {
            const float4 Lm = ldg4(pv.lamlog + eo);
            const float ax = K4.x * expf(lp4.x - Lm.x), ay = K4.y * expf(lp4.y - Lm.y);
            const float az = K4.z * expf(lp4.z - Lm.z), aw = K4.w * expf(lp4.w - Lm.w);
            ck = warp_sum(fmaf(ax, k4.x, fmaf(ay, k4.y, fmaf(az, k4.z, aw * k4.w))));
            cq = warp_sum(fmaf(ax, q4.x, fmaf(ay, q4.y, fmaf(az, q4.z, aw * q4.w))));
        } else {
            const float g = expf(lp4.x - __ldg(pv.lamlog + e0 + l));
            ck = warp_sum(fmaf(K4.x, k4.x, fmaf(K4.y, k4.y, fmaf(K4.z, k4.z, K4.w * k4.w)))) * g;
            cq = warp_sum(fmaf(K4.x, q4.x, fmaf(K4.y, q4.y, fmaf(K4.z, q4.z, K4.w * q4.w)))) * g;
        }
        r4 = make_float4(fmaf(ck, U4.x, r4.x), fmaf(ck, U4.y, r4.y), fmaf(ck, U4.z, r4.z),
                         fmaf(ck, U4.w, r4.w));
        y4 = make_float4(fmaf(cq, U4.x, y4.x), fmaf(cq, U4.y, y4.y), fmaf(cq, U4.z, y4.z),
                         fmaf(cq, U4.w, y4.w));
    }

    // ---- delta correction and output -----------------------------------------
    const float4 u4 = make_float4(beta * (v4.x - r4.x), beta * (v4.y - r4.y),
                                  beta * (v4.z - r4.z), beta * (v4.w - r4.w));
    st4(a.y + ro, make_float4(fmaf(kq, u4.x, y4.x), fmaf(kq, u4.y, y4.y), fmaf(kq, u4.z, y4.z),
                              fmaf(kq, u4.w, y4.w)));

    // ---- append entry L -------------------------------------------------------
    {
        const size_t eo = (e0 + L) * kD + 4 * lane;
        st4(pv.klog + eo, k4);
        st4(pv.ulog + eo, u4);
        if constexpr (PER_KEY) st4(pv.lamlog + eo, lp4);
        else if (lane == 0) pv.lamlog[e0 + L] = lp4.x;
    }
    if (L + 1 < W) {
        if constexpr (PER_KEY) st4(pv.lbar + hd * kD + 4 * lane, lp4);
        else if (lane == 0) pv.lbar[hd] = lp4.x;
        if (lane == 0) pv.len[hd] = L + 1;
        return;
    }
    // ---- window end: fold the W entries into the base, start a new window ----
    __syncwarp();
    fold_warp<INT8, PER_KEY, kFoldCommit>(pv, hd, L + 1, lp_s[warp], lp4.x, nullptr, lane);
    if constexpr (PER_KEY) st4(pv.lbar + hd * kD + 4 * lane, make_float4(0.f, 0.f, 0.f, 0.f));
    else if (lane == 0) pv.lbar[hd] = 0.0f;
    if (lane == 0) pv.len[hd] = 0;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
}

}  // namespace

cudaError_t prepare_step_kernels() {
    cudaError_t e;
    if ((e = set_smem(eager_step_kernel<false>, eager_smem_bytes())) != cudaSuccess) return e;
    if ((e = set_smem(eager_step_kernel<true>, eager_smem_bytes())) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_eager_step(const StepArgs& a, bool per_key, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.batch) * static_cast<unsigned>(a.pv.H));
    if (per_key)
        eager_step_kernel<true><<<grid, kThreads, eager_smem_bytes(), s>>>(a);
    else
        eager_step_kernel<false><<<grid, kThreads, eager_smem_bytes(), s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_log_step(const StepArgs& a, bool int8, bool per_key, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.batch) * a.pv.H;
    const dim3 grid(static_cast<unsigned>((rows + kWarps - 1) / kWarps));
    if (int8) {
        if (per_key)
            log_step_kernel<true, true><<<grid, kThreads, 0, s>>>(a);
        else
            log_step_kernel<true, false><<<grid, kThreads, 0, s>>>(a);
    } else {
        if (per_key)
            log_step_kernel<false, true><<<grid, kThreads, 0, s>>>(a);
        else
            log_step_kernel<false, false><<<grid, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace ls
