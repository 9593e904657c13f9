// ls_fold.cu -- window commit and logical read of libls (sm_103a).
//
// Deferred / INT8: one CTA per (slot, head) folds the live log into the base
// (ls_window_commit: "DeltaLog: Deferred Materialization of Recurrent States
// for Linear Attention Decoding", §3.1 merge without a new token; INT8 window
// closed early and requantized, "LeapQuant: Efficient Linear Attention with
// Accurate Recurrent State Quantization", §3.2 eq. 4) or into a caller buffer
// (ls_pool_read: DeltaLog §3.2 eq. 7, the logical state), with the same
// CTA-cooperative fold the decode step uses at a window's end (ls_warp.cuh).
// Eager: the logical state is the dense base; ls_pool_read transposes its
// S^T tiles back to [d_k][d_v].
#include <cuda_runtime.h>

#include "ls_device.cuh"
#include "ls_internal.cuh"
#include "ls_warp.cuh"

namespace ls {

namespace {

template <bool INT8, bool PER_KEY, int MODE, bool COMP>
__global__ void __launch_bounds__(kThreads, 2) fold_kernel(const AuxArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    const int slot = __ldg(a.slots + n);
    if (slot < 0 || slot >= pv.P) {
        if (threadIdx.x == 0) flag_status(pv.status, kDevSlotRange);
        return;
    }
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const int L = pv.len[hd];
    if (L < 0 || L >= pv.cap) {
        if (threadIdx.x == 0) flag_status(pv.status, kDevBadState);
        return;
    }
    if (MODE == kFoldCommit && L <= pv.R) return;  // already at a boundary (only the pairs)
    const FoldSmem fs = fold_smem(smem, INT8);
    if (threadIdx.x == 0) {
        mbar_init(fs.bar, 1);
        mbar_init(fs.lbar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    // per-key gate: lbar is read row by row from global memory by the fold
    // (it is reset only after the fold); scalar gate: one value
    const float lb = PER_KEY ? 0.0f : pv.lbar[hd];
    float* out = nullptr;
    if constexpr (MODE == kFoldRead) out = a.state_out + (static_cast<size_t>(n) * H + h) * (kD * kD);
    const TokenIn none{nullptr, nullptr, nullptr, nullptr, 0.0f, nullptr, 0};
    FoldPipe pp;
    const bool ok = fold_cta<INT8, PER_KEY, MODE, COMP>(pv, hd, L, pv.lbar + hd * (PER_KEY ? kD : 1), lb,
                                                  out, fs, pp, none, -1, 0);
    if (MODE == kFoldCommit && ok) {
        __syncthreads();  // every reader of lbar is done
        if (PER_KEY) {
            if (threadIdx.x < kD / 4) st4(pv.lbar + hd * kD + 4 * threadIdx.x, make_float4(0.f, 0.f, 0.f, 0.f));
        } else if (threadIdx.x == 0) {
            pv.lbar[hd] = 0.0f;
        }
        if (threadIdx.x == 0) pv.len[hd] = pv.R;
    }
}

// Eager base S^T [j][i] -> logical out[i][j].
__global__ void __launch_bounds__(kThreads) eager_read_kernel(const AuxArgs a) {
    extern __shared__ __align__(16) float tsm[];  // [128][129]
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    const int slot = __ldg(a.slots + n);
    if (slot < 0 || slot >= pv.P) {
        if (threadIdx.x == 0) flag_status(pv.status, kDevSlotRange);
        return;
    }
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const float* base = reinterpret_cast<const float*>(pv.base) + hd * (kD * kD);
    for (int idx = threadIdx.x; idx < kD * kD; idx += kThreads) {
        const int j = idx >> 7, i = idx & (kD - 1);
        tsm[i * (kD + 1) + j] = base[idx];
    }
    __syncthreads();
    float* out = a.state_out + (static_cast<size_t>(n) * H + h) * (kD * kD);
    for (int idx = threadIdx.x; idx < kD * kD; idx += kThreads) {
        const int i = idx >> 7, j = idx & (kD - 1);
        out[idx] = tsm[i * (kD + 1) + j];
    }
}

template <bool INT8, bool PER_KEY>
cudaError_t launch_mode(const AuxArgs& a, bool commit, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    const size_t sm = fold_smem_bytes(INT8);
    if (commit && INT8 && a.pv.R > 0)
        fold_kernel<INT8, PER_KEY, kFoldCommit, INT8><<<grid, kThreads, sm, s>>>(a);
    else if (commit)
        fold_kernel<INT8, PER_KEY, kFoldCommit, false><<<grid, kThreads, sm, s>>>(a);
    else
        fold_kernel<INT8, PER_KEY, kFoldRead, false><<<grid, kThreads, sm, s>>>(a);
    return cudaGetLastError();
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
}

template <bool INT8, bool PER_KEY>
cudaError_t prepare_mode() {
    cudaError_t e = set_smem(fold_kernel<INT8, PER_KEY, kFoldCommit, false>, fold_smem_bytes(INT8));
    if (e != cudaSuccess) return e;
    if ((e = set_smem(fold_kernel<INT8, PER_KEY, kFoldCommit, INT8>, fold_smem_bytes(INT8))) != cudaSuccess)
        return e;
    return set_smem(fold_kernel<INT8, PER_KEY, kFoldRead, false>, fold_smem_bytes(INT8));
}

}  // namespace

cudaError_t launch_fold(const AuxArgs& a, bool int8, bool per_key, bool commit, cudaStream_t s) {
    if (int8)
        return per_key ? launch_mode<true, true>(a, commit, s) : launch_mode<true, false>(a, commit, s);
    return per_key ? launch_mode<false, true>(a, commit, s) : launch_mode<false, false>(a, commit, s);
}

cudaError_t launch_eager_read(const AuxArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    eager_read_kernel<<<grid, kThreads, transpose_smem_bytes(), s>>>(a);
    return cudaGetLastError();
}

cudaError_t prepare_fold_kernels() {
    cudaError_t e;
    if ((e = prepare_mode<false, false>()) != cudaSuccess) return e;
    if ((e = prepare_mode<false, true>()) != cudaSuccess) return e;
    if ((e = prepare_mode<true, false>()) != cudaSuccess) return e;
    if ((e = prepare_mode<true, true>()) != cudaSuccess) return e;
    return set_smem(eager_read_kernel, transpose_smem_bytes());
}

}  // namespace ls
