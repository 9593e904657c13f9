// ls_eager.cu -- eager FP32 decode-step kernel of libls (sm_103a).
//
// One CTA of 256 threads decodes one (request, head) per token.  The head's
// dense state (S^T: 128 value columns x 128 key rows, FP32, 64 KiB) is staged
// in shared memory by four 1-D bulk asynchronous copies (TMA, cp.async.bulk)
// of one quarter (32 columns) each, completing on four mbarriers; the warps
// consume quarter r as soon as it lands.  Each value column is reduced over
// the 128 key rows by a group of 8 lanes (16 rows per lane, 3 shuffle
// levels) -- the two GEMVs r = S^T(alpha.k), y0 = S^T(alpha.q) of the
// delta-rule step -- and written back in place.  Value columns are
// independent, so no CTA waits on another.
//
// Page: "LeapQuant: Efficient Linear Attention with Accurate Recurrent State
// Quantization", App. A (GDN / KDA recurrences) with eq. 1.
#include <cuda_runtime.h>

#include "ls_device.cuh"
#include "ls_internal.cuh"

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
// eager FP32: read S, r = S^T(alpha.k), u = beta (v - r),
//     S <- Diag(alpha) S + k u^T (written in place), y = S^T(alpha.q) + (k.q) u
//     (= S_t^T q).  LeapQuant App. A with eq. 1.
// ---------------------------------------------------------------------------
template <bool PER_KEY>
__global__ void __launch_bounds__(kThreads, 3) eager_step_kernel(const StepArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    pdl_enter();
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
    gather16(xk_s, g, xk);
    gather16(xq_s, g, xq);

#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
        const int j = round_col(r, warp, c);
        if (!wait_quarter(bars, r, a.pv.status)) return;
        float s[16];
        load_tile16(tile, j, g, s);
        float rr = 0.0f, yy = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            rr = fmaf(s[e], xk[e], rr);
            yy = fmaf(s[e], xq[e], yy);
        }
        rr = group8_sum(rr);
        yy = group8_sum(yy);
        const float u = a.pv.plain ? v_s[j] : beta * (v_s[j] - rr);
        if (g == 0) y_s[j] = fmaf(kq, u, yy);
        float* dst = gtile + j * kD;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int i0 = run_row(g, m);
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

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
}

}  // namespace

cudaError_t prepare_eager_step_kernels() {
    cudaError_t e;
    if ((e = set_smem(eager_step_kernel<false>, eager_smem_bytes())) != cudaSuccess) return e;
    return set_smem(eager_step_kernel<true>, eager_smem_bytes());
}

cudaError_t launch_eager_step(const StepArgs& a, bool per_key, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.batch) * static_cast<unsigned>(a.pv.H));
    return launch_dependent(per_key ? eager_step_kernel<true> : eager_step_kernel<false>, grid,
                            eager_smem_bytes(), s, a);
}

}  // namespace ls
