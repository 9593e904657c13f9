// ls_aux.cu -- slot lifecycle kernels of libls (sm_103a): load a dense state
// into a slot (quantizing it for the INT8 variant), reset slots, and read
// back INT8 codes and log metadata.  A fresh slot takes its prefill state and
// an empty log; a reused slot is cleared ("DeltaLog: Deferred Materialization
// of Recurrent States for Linear Attention Decoding", §4, state-slot
// lifecycle).  None of these is on the per-token path.
#include <cuda_runtime.h>

#include "ls_device.cuh"
#include "ls_internal.cuh"
#include "ls_warp.cuh"

namespace ls {

namespace {

constexpr int kPad = kD + 1;  // padded row stride of a transposed tile

__device__ __forceinline__ bool slot_of(const AuxArgs& a, int n, int* slot) {
    const int s = __ldg(a.slots + n);
    if (s < 0 || s >= a.pv.P) {
        if (threadIdx.x == 0) flag_status(a.pv.status, kDevSlotRange);
        return false;
    }
    *slot = s;
    return true;
}

__device__ __forceinline__ void clear_log(const PoolView& pv, size_t hd) {
    if (pv.lbar == nullptr) return;
    if (pv.dl == kD) {
        if (threadIdx.x < kD) pv.lbar[hd * kD + threadIdx.x] = 0.0f;
    } else if (threadIdx.x == 0) {
        pv.lbar[hd] = 0.0f;
    }
    if (threadIdx.x == 0) pv.len[hd] = 0;
}

// Eager: state_in[n][h] (logical [i][j]) -> base S^T [j][i].
__global__ void __launch_bounds__(kThreads) load_eager_kernel(const AuxArgs a) {
    extern __shared__ __align__(16) float t[];  // [128][129] = S[i][j]
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const float* in = a.state_in + (static_cast<size_t>(n) * H + h) * (kD * kD);
    for (int idx = threadIdx.x; idx < kD * kD; idx += kThreads) {
        const int i = idx >> 7, j = idx & (kD - 1);
        t[i * kPad + j] = in[idx];
    }
    __syncthreads();
    float* base = reinterpret_cast<float*>(pv.base) + hd * (kD * kD);
    for (int idx = threadIdx.x; idx < kD * kD; idx += kThreads) {
        const int j = idx >> 7, i = idx & (kD - 1);
        base[idx] = t[i * kPad + j];
    }
}

// Deferred / INT8: state_in[n][h] -> base [i][j]; INT8 quantizes every key
// row with its own scale (the rule of a window end).  Warp w takes rows
// w, w + 8, ...; lane l columns 4l..4l+3.
template <bool INT8>
__global__ void __launch_bounds__(kThreads) load_rows_kernel(const AuxArgs a) {
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const float* in = a.state_in + (static_cast<size_t>(n) * H + h) * (kD * kD);
    for (int i = warp; i < kD; i += kWarps) {
        const float4 v = ldg4(in + i * kD + 4 * lane);
        if constexpr (!INT8) {
            st4(reinterpret_cast<float*>(pv.base) + hd * (kD * kD) + i * kD + 4 * lane, v);
        } else {
            float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
            m = warp_max(m);
            const float s = __fdiv_rn(m, 127.0f);
            reinterpret_cast<uint32_t*>(pv.base)[hd * (kD * kD / 4) + i * (kD / 4) + lane] =
                pack_codes4(v, s);
            if (lane == 0) pv.scale[hd * kD + i] = s;
        }
    }
    clear_log(pv, hd);
}

template <bool INT8>
__global__ void __launch_bounds__(kThreads) reset_kernel(const AuxArgs a) {
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    float4* base = reinterpret_cast<float4*>(reinterpret_cast<unsigned char*>(pv.base) +
                                             hd * tile_bytes(INT8));
    const int n4 = static_cast<int>(tile_bytes(INT8) / 16);
    for (int idx = threadIdx.x; idx < n4; idx += kThreads) base[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (INT8) {
        if (threadIdx.x < kD) pv.scale[hd * kD + threadIdx.x] = 0.0f;
    }
    clear_log(pv, hd);
}

// INT8 codes (already [i][j]) and scales of n slots.
__global__ void __launch_bounds__(kThreads) read_int8_kernel(const AuxArgs a) {
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const size_t o = static_cast<size_t>(n) * H + h;
    const int4* src = reinterpret_cast<const int4*>(reinterpret_cast<const int8_t*>(pv.base) +
                                                    hd * (kD * kD));
    int4* dst = reinterpret_cast<int4*>(a.codes_out + o * (kD * kD));
    for (int idx = threadIdx.x; idx < kD * kD / 16; idx += kThreads) dst[idx] = src[idx];
    if (threadIdx.x < kD) a.scales_out[o * kD + threadIdx.x] = pv.scale[hd * kD + threadIdx.x];
}

__global__ void __launch_bounds__(128) read_log_meta_kernel(const AuxArgs a) {
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const size_t o = static_cast<size_t>(n) * H + h;
    if (threadIdx.x == 0) a.len_out[o] = pv.len[hd];
    if (a.lbar_out != nullptr && threadIdx.x < pv.dl)
        a.lbar_out[o * pv.dl + threadIdx.x] = pv.lbar[hd * pv.dl + threadIdx.x];
}

}  // namespace

cudaError_t prepare_aux_kernels() {
    return cudaFuncSetAttribute(load_eager_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(transpose_smem_bytes()));
}

cudaError_t launch_load(const AuxArgs& a, bool int8, bool has_log, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    if (!has_log)
        load_eager_kernel<<<grid, kThreads, transpose_smem_bytes(), s>>>(a);
    else if (int8)
        load_rows_kernel<true><<<grid, kThreads, 0, s>>>(a);
    else
        load_rows_kernel<false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_reset(const AuxArgs& a, bool int8, bool /*has_log*/, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    if (int8)
        reset_kernel<true><<<grid, kThreads, 0, s>>>(a);
    else
        reset_kernel<false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_read_int8(const AuxArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    read_int8_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_read_log_meta(const AuxArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    read_log_meta_kernel<<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ls
