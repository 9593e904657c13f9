// ls_device.cuh -- device helpers of libls: bulk asynchronous copies with
// mbarrier completion (sm_90+ / sm_103a), bounded waits, warp reductions,
// the INT8 rounding rule, and the eager kernel's thread <-> tile mapping.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ls_internal.cuh"

namespace ls {

// ---- mbarrier + cp.async.bulk (1-D TMA) -----------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Invalidate a barrier whose phases are all complete, before its memory is
// used for anything else.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Make the initialised barriers visible to the asynchronous proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy completing `bytes` transactions on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before its
// later asynchronous-proxy ones (a bulk copy refilling a stage just read).
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Iteration limit of every wait on an mbarrier.  A bulk copy from valid
// memory completes in microseconds; the limit only keeps a kernel from
// spinning forever if something went wrong.
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    for (uint32_t it = 0; it < kWaitLimit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---- loads / stores --------------------------------------------------------

__device__ __forceinline__ float4 ldg4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}
// Streaming load (read once, do not keep in L1).
__device__ __forceinline__ float4 ld_stream4(const float* p) {
    float4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ void st4(float* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
}

// ---- reductions -------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
// max over the warp's 32 lanes of |x| (one redux; NaN inputs are ignored).
__device__ __forceinline__ float warp_absmax_redux(float x) {
    float r;
    asm volatile("redux.sync.max.abs.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
    return r;
}

// Sum over the 8 lanes of a lane group (lanes that differ in bits 0..2).
__device__ __forceinline__ float group8_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}

// ---- eager tile mapping -------------------------------------------------------
// The eager kernel stages a head's S^T tile (value column j = 128 contiguous
// key rows, 512 B) in shared memory.  Each value column is owned by a group of
// 8 lanes (g = lane & 7 picks the rows, c = lane >> 3 the column inside the
// warp's 4 columns); round r (0..3) of warp w covers column j = 32 r + 4 w + c.
// Lane g owns the 16 key rows 32 m + 4 g + (0..3), m = 0..3, so a quarter warp
// reads 128 contiguous bytes of one column.
__device__ __forceinline__ int run_row(int g, int m) { return 32 * m + 4 * g; }
__device__ __forceinline__ int round_col(int r, int warp, int c) { return 32 * r + 4 * warp + c; }

// The 16 tile values a lane owns in column j.
__device__ __forceinline__ void load_tile16(const unsigned char* tile, int j, int g, float (&s)[16]) {
    const float* t = reinterpret_cast<const float*>(tile) + j * kD;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 v = *reinterpret_cast<const float4*>(t + 32 * m + 4 * g);
        s[4 * m + 0] = v.x;
        s[4 * m + 1] = v.y;
        s[4 * m + 2] = v.z;
        s[4 * m + 3] = v.w;
    }
}

// Per-lane copy of a 128-vector at the lane's 16 rows.
__device__ __forceinline__ void gather16(const float* vec, int g, float (&x)[16]) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 v = *reinterpret_cast<const float4*>(vec + run_row(g, m));
        x[4 * m + 0] = v.x;
        x[4 * m + 1] = v.y;
        x[4 * m + 2] = v.z;
        x[4 * m + 3] = v.w;
    }
}

// Per-key-row INT8 parameters from the row's absmax B: stored scale
// s = B / 127 and quantization factor f = 127 / B (correctly rounded FP32;
// LeapQuant App. B.3 writes dequant = (Z / 127) B).  A row whose scale or
// factor is not a positive finite FP32 number gets s = f = 0 (codes 0).
__device__ __forceinline__ void row_quant_params(float amax, float& s, float& f) {
    s = __fdiv_rn(amax, 127.0f);
    f = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    if (!(s > 0.0f) || !(f <= 3.402823466e38f)) {
        s = 0.0f;
        f = 0.0f;
    }
}

// Programmatic dependent launch: let the next kernel on the stream be
// scheduled as soon as every CTA of this one has started, then wait until
// the previous kernel has completed and its memory is visible.  Called first
// thing in a step kernel, before any global memory access; a no-op when the
// launch carries no programmatic dependency.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Four bfloat16 (two words, low half first) widened to FP32, exactly.
__device__ __forceinline__ float4 bf16x4_to_float4(uint2 w) {
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

// FP32 -> bfloat16, round to nearest even, four at a time.
__device__ __forceinline__ uint2 float4_to_bf16x4(float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// Four binary16 (two words, low half first) widened to FP32, exactly.
__device__ __forceinline__ float4 half4_to_float4(uint2 w) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// FP32 -> binary16, round to nearest even, four at a time.
__device__ __forceinline__ uint2 float4_to_half4(float4 v) {
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// One stored 16-bit key factor widened to FP32: bfloat16 (bf16) or binary16.
__device__ __forceinline__ float key16_to_float(unsigned short h, bool bf16) {
    return bf16 ? __uint_as_float(static_cast<uint32_t>(h) << 16) : __half2float(__ushort_as_half(h));
}

// Four stored key factors (16-byte or 8-byte group at element index e, a
// multiple of 4) as FP32: FP32, bfloat16 (k16) or binary16 (rec16).
__device__ __forceinline__ float4 key4_at(const void* p, size_t e, const PoolView& pv) {
    if (pv.k16) return bf16x4_to_float4(reinterpret_cast<const uint2*>(p)[e >> 2]);
    if (pv.rec16) return half4_to_float4(reinterpret_cast<const uint2*>(p)[e >> 2]);
    return reinterpret_cast<const float4*>(p)[e >> 2];
}

// The same for value factors: FP32 or binary16 (rec16).
__device__ __forceinline__ float4 val4_at(const void* p, size_t e, const PoolView& pv) {
    if (pv.rec16) return half4_to_float4(reinterpret_cast<const uint2*>(p)[e >> 2]);
    return reinterpret_cast<const float4*>(p)[e >> 2];
}

// Bytes per stored key / value factor.
__host__ __device__ __forceinline__ uint32_t key_bytes(const PoolView& pv) {
    return (pv.k16 || pv.rec16) ? 2u : 4u;
}
__host__ __device__ __forceinline__ uint32_t val_bytes(const PoolView& pv) { return pv.rec16 ? 2u : 4u; }

// exp(d) of a replay decay d = lp - Lambda_l <= 0 (per-key gate: four per lane
// and log entry), by the hardware exponential: relative error about 2^-21
// plus |d| 2^-24, with |d| at most a window's cumulative log-decay, far inside
// the FP32 tolerance of the readouts.  Every replay of a log entry (the fused
// step kernels and the split-replay prepare kernel) uses this one function,
// so the split and fused paths stay bit-identical.
__device__ __forceinline__ float replay_decay(float d) { return __expf(d); }

// Log record formats, a template parameter of the step kernels so that the
// per-entry replay carries no format branches: FP32 key and value factors,
// bfloat16 keys (DeltaLog §3.4), or binary16 keys and values (LeapQuant
// §4.1, §4.3).  The pool view's k16 / rec16 select the instantiation.
constexpr int kRecFP32 = 0, kRecBF16K = 1, kRecFP16 = 2;
__host__ __device__ constexpr uint32_t rec_key_bytes(int rec) { return rec == kRecFP32 ? 4u : 2u; }
__host__ __device__ constexpr uint32_t rec_val_bytes(int rec) { return rec == kRecFP16 ? 2u : 4u; }

template <int REC>
__device__ __forceinline__ float4 rec_key4(const void* p, size_t e) {
    if constexpr (REC == kRecBF16K) return bf16x4_to_float4(reinterpret_cast<const uint2*>(p)[e >> 2]);
    else if constexpr (REC == kRecFP16) return half4_to_float4(reinterpret_cast<const uint2*>(p)[e >> 2]);
    else return reinterpret_cast<const float4*>(p)[e >> 2];
}
template <int REC>
__device__ __forceinline__ float4 rec_val4(const void* p, size_t e) {
    if constexpr (REC == kRecFP16) return half4_to_float4(reinterpret_cast<const uint2*>(p)[e >> 2]);
    else return reinterpret_cast<const float4*>(p)[e >> 2];
}

// Hint: bring the 128-byte line holding p into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void flag_status(int32_t* status, int32_t bit) {
    atomicOr(status, bit);
}

}  // namespace ls
