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

// Deferred / INT8: state_in[n][h] -> base; INT8 quantizes every key row with
// its own scale (the rule of a window end).  Warp w takes the 4-row groups
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
    for (int i4 = warp; i4 < kD / 4; i4 += kWarps) {
        float4 v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = ldg4(in + (4 * i4 + m) * kD + 4 * lane);
        if constexpr (!INT8) {
#pragma unroll
            for (int m = 0; m < 4; ++m)
                st4(reinterpret_cast<float*>(pv.base) + hd * (kD * kD) + (4 * i4 + m) * kD + 4 * lane,
                    v[m]);
        } else {
            float f[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                float mx = fmaxf(fmaxf(fabsf(v[m].x), fabsf(v[m].y)), fmaxf(fabsf(v[m].z), fabsf(v[m].w)));
                mx = warp_max(mx);
                float sc;
                row_quant_params(mx, sc, f[m]);
                if (lane == 0) pv.scale[hd * kD + 4 * i4 + m] = sc;
            }
            float2 lo[4], hi[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                lo[m] = make_float2(v[m].x, v[m].y);
                hi[m] = make_float2(v[m].z, v[m].w);
            }
            reinterpret_cast<uint4*>(pv.base)[quad_index(hd, i4, lane)] = pack_quad(lo, hi, 0, f);
        }
    }
    clear_log(pv, hd);
}

// INT8, smoothed per-value-column format: state_in[n][h] -> codes, smoothing
// factors c and column scales b, with the window end's own quantization
// ("LeapQuant: Efficient Linear Attention with Accurate Recurrent State
// Quantization", §3.4 eq. 7); warp w holds key rows 16w..16w+15.
__global__ void __launch_bounds__(kThreads) load_cols_kernel(const AuxArgs a) {
    __shared__ __align__(16) float red[kWarps * kD];
    __shared__ __align__(16) float fcol[kD];
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;  // uniform over the CTA
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const float* in = a.state_in + (static_cast<size_t>(n) * H + h) * (kD * kD);
    float2 lo[16], hi[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float4 v = ldg4(in + (16 * warp + r) * kD + 4 * lane);
        lo[r] = make_float2(v.x, v.y);
        hi[r] = make_float2(v.z, v.w);
    }
    quantize_cols_cta(lo, hi, pv.base, hd, pv.scale + hd * kD, pv.colf + hd * kD, red, fcol);
    clear_log(pv, hd);
}

// INT8 with compensator pairs: state_in[n][h] -> pairs fitted from a cold
// start, then the residual in the pool's format, and a log that holds only
// the pairs ("LeapQuant: Efficient Linear Attention with Accurate Recurrent
// State Quantization", §3.3 eq. 5-6); warp w holds key rows 16w..16w+15.
__global__ void __launch_bounds__(kThreads) load_comp_kernel(const AuxArgs a) {
    __shared__ __align__(16) float red[kWarps * kD];
    __shared__ __align__(16) float vs[kD], ws[kD], ks[kD];
    __shared__ float nz[4];
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;  // uniform over the CTA
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const float* in = a.state_in + (static_cast<size_t>(n) * H + h) * (kD * kD);
    float2 lo[16], hi[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float4 v = ldg4(in + (16 * warp + r) * kD + 4 * lane);
        lo[r] = make_float2(v.x, v.y);
        hi[r] = make_float2(v.z, v.w);
    }
    fit_compensators_cta(lo, hi, pv, hd, vs, ws, ks, red, nz);
    if (pv.colf != nullptr)
        quantize_cols_cta(lo, hi, pv.base, hd, pv.scale + hd * kD, pv.colf + hd * kD, red, vs);
    else
        quantize_rows_cta(lo, hi, pv.base, hd, pv.scale + hd * kD);
    if (pv.dl == kD) {
        if (threadIdx.x < kD) pv.lbar[hd * kD + threadIdx.x] = 0.0f;
    } else if (threadIdx.x == 0) {
        pv.lbar[hd] = 0.0f;
    }
    if (threadIdx.x == 0) pv.len[hd] = pv.R;
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
        // a zero state: per-row scales 0, or (column-scale format) floored
        // smoothing factors and zero column scales
        if (threadIdx.x < kD) {
            pv.scale[hd * kD + threadIdx.x] = pv.colf != nullptr ? kSmoothFloor : 0.0f;
            if (pv.colf != nullptr) pv.colf[hd * kD + threadIdx.x] = 0.0f;
        }
    }
    clear_log(pv, hd);
    if (INT8 && pv.R > 0) {
        // a zero state's pairs: k~ = 0, u~ = the cold start 1 / sqrt(128)
        const size_t kb = hd * static_cast<size_t>(pv.cap);
        for (int idx = threadIdx.x; idx < pv.R * kD; idx += kThreads) {
            if (pv.rec16) {
                reinterpret_cast<__half*>(pv.klog)[kb * kD + idx] = __float2half_rn(0.0f);
                reinterpret_cast<__half*>(pv.ulog)[kb * kD + idx] = __float2half_rn(0.08838834764831845f);
            } else {
                pv.klog[kb * kD + idx] = 0.0f;
                pv.ulog[kb * kD + idx] = 0.08838834764831845f;
            }
        }
        const int nl = pv.dl == kD ? pv.R * kD : pv.R;
        for (int idx = threadIdx.x; idx < nl; idx += kThreads)
            pv.lamlog[hd * static_cast<size_t>(pv.lam_stride) + idx] = 0.0f;
        __syncthreads();  // clear_log's len = 0 store is ordered before this one
        if (threadIdx.x == 0) pv.len[hd] = pv.R;
    }
}

// INT8 codes in the logical layout codes[n][h][i][j] and scales[n][h][i].
__global__ void __launch_bounds__(kThreads) read_int8_kernel(const AuxArgs a) {
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const size_t o = static_cast<size_t>(n) * H + h;
    uint32_t* codes = reinterpret_cast<uint32_t*>(a.codes_out + o * (kD * kD));
    for (int i4 = warp; i4 < kD / 4; i4 += kWarps) {
        const uint4 w = reinterpret_cast<const uint4*>(pv.base)[quad_index(hd, i4, lane)];
        // row r of the quad: byte r of each column word
        const uint32_t lo01 = __byte_perm(w.x, w.y, 0x5140), hi01 = __byte_perm(w.x, w.y, 0x7362);
        const uint32_t lo23 = __byte_perm(w.z, w.w, 0x5140), hi23 = __byte_perm(w.z, w.w, 0x7362);
        codes[(4 * i4 + 0) * (kD / 4) + lane] = __byte_perm(lo01, lo23, 0x5410);
        codes[(4 * i4 + 1) * (kD / 4) + lane] = __byte_perm(lo01, lo23, 0x7632);
        codes[(4 * i4 + 2) * (kD / 4) + lane] = __byte_perm(hi01, hi23, 0x5410);
        codes[(4 * i4 + 3) * (kD / 4) + lane] = __byte_perm(hi01, hi23, 0x7632);
    }
    if (threadIdx.x < kD) a.scales_out[o * kD + threadIdx.x] = pv.scale[hd * kD + threadIdx.x];
}

__global__ void __launch_bounds__(128) read_colf_kernel(const AuxArgs a) {
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const size_t o = static_cast<size_t>(n) * H + h;
    a.scales_out[o * kD + threadIdx.x] = pv.colf[hd * kD + threadIdx.x];
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
    else if (int8 && a.pv.R > 0)
        load_comp_kernel<<<grid, kThreads, 0, s>>>(a);
    else if (int8 && a.pv.colf != nullptr)
        load_cols_kernel<<<grid, kThreads, 0, s>>>(a);
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

cudaError_t launch_read_colf(const AuxArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    read_colf_kernel<<<grid, kD, 0, s>>>(a);
    return cudaGetLastError();
}

// The current pairs: k_out [n][H][R][d_k] (state_out), u_out [n][H][R][d_v]
// (scales_out).
__global__ void __launch_bounds__(kThreads) read_comp_kernel(const AuxArgs a) {
    const PoolView& pv = a.pv;
    const int H = pv.H;
    const int n = blockIdx.x / H, h = blockIdx.x - n * H;
    int slot;
    if (!slot_of(a, n, &slot)) return;
    const size_t hd = static_cast<size_t>(slot) * H + h;
    const size_t o = (static_cast<size_t>(n) * H + h) * static_cast<size_t>(pv.R) * kD;
    const size_t kb = hd * static_cast<size_t>(pv.cap) * kD;
    for (int idx = threadIdx.x; idx < pv.R * kD; idx += kThreads) {
        if (pv.rec16) {
            a.state_out[o + idx] = __half2float(reinterpret_cast<const __half*>(pv.klog)[kb + idx]);
            a.scales_out[o + idx] = __half2float(reinterpret_cast<const __half*>(pv.ulog)[kb + idx]);
        } else {
            a.state_out[o + idx] = pv.klog[kb + idx];
            a.scales_out[o + idx] = pv.ulog[kb + idx];
        }
    }
}

// A new pool's states as a reset leaves them: for compensator pools every
// log starts with the zero state's pairs (k~ = 0, u~ = 1 / sqrt(128),
// snapshot 0), so len = R.  One CTA per state; the memory is zeroed before.
__global__ void __launch_bounds__(kD) init_comp_kernel(const PoolView pv) {
    const size_t hd = blockIdx.x;
    const size_t kb = hd * static_cast<size_t>(pv.cap) * kD;
    for (int idx = threadIdx.x; idx < pv.R * kD; idx += kD) {
        if (pv.rec16)
            reinterpret_cast<__half*>(pv.ulog)[kb + idx] = __float2half_rn(0.08838834764831845f);
        else
            pv.ulog[kb + idx] = 0.08838834764831845f;
    }
    if (threadIdx.x == 0) pv.len[hd] = pv.R;
}

cudaError_t launch_init_comp(const PoolView& pv, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(pv.P) * static_cast<unsigned>(pv.H));
    init_comp_kernel<<<grid, kD, 0, s>>>(pv);
    return cudaGetLastError();
}

cudaError_t launch_read_comp(const AuxArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    read_comp_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

// LS_CHECK_SLOTS: one CTA counts every in-range slot of a slot list in
// pv.mark, flags a count above one, and clears the counts for the next call.
// Slots out of range are left to the call that follows, which flags them.
__global__ void __launch_bounds__(1024) slot_check_kernel(const PoolView pv, const int32_t* slots, int32_t n) {
    for (int b = threadIdx.x; b < n; b += blockDim.x) {
        const int s = __ldg(slots + b);
        if (s >= 0 && s < pv.P) atomicAdd(pv.mark + s, 1);
    }
    __syncthreads();
    bool dup = false;
    for (int b = threadIdx.x; b < n; b += blockDim.x) {
        const int s = __ldg(slots + b);
        if (s >= 0 && s < pv.P && __ldcg(pv.mark + s) > 1) dup = true;
    }
    if (__syncthreads_or(dup) && threadIdx.x == 0) flag_status(pv.status, kDevSlotDup);
    for (int b = threadIdx.x; b < n; b += blockDim.x) {
        const int s = __ldg(slots + b);
        if (s >= 0 && s < pv.P) pv.mark[s] = 0;
    }
}

cudaError_t launch_slot_check(const PoolView& pv, const int32_t* slots, int32_t n, cudaStream_t s) {
    slot_check_kernel<<<1, 1024, 0, s>>>(pv, slots, n);
    return cudaGetLastError();
}

cudaError_t launch_read_log_meta(const AuxArgs& a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.n) * static_cast<unsigned>(a.pv.H));
    read_log_meta_kernel<<<grid, 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ls
