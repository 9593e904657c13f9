// ls_warp.cuh -- warp-per-head building blocks of the deferred and per-window
// INT8 variants (sm_103a).
//
// One warp owns one (slot, head).  The base is stored row-major, S[i][j]
// (key row i, value column j); lane l owns value columns 4l..4l+3 and, for
// vectors indexed by key, key rows 4l..4l+3.  A base row is one coalesced
// warp access (512 B FP32, 128 B INT8), so the GEMVs S^T x reduce over key
// rows inside each lane, with no cross-lane reduction, and a key row's absmax
// (the INT8 scale) is a warp reduction.
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

// 4 INT8 codes (one 32-bit word, little-endian) -> 4 floats.
__device__ __forceinline__ float4 codes4(uint32_t w) {
    return make_float4(static_cast<float>(static_cast<int8_t>(w & 0xffu)),
                       static_cast<float>(static_cast<int8_t>((w >> 8) & 0xffu)),
                       static_cast<float>(static_cast<int8_t>((w >> 16) & 0xffu)),
                       static_cast<float>(static_cast<int8_t>(w >> 24)));
}

template <bool INT8>
struct BaseRows {
    // Row i of head hd, the lane's 4 columns.
    static __device__ __forceinline__ float4 stream(const void* base, size_t hd, int i, int lane) {
        if constexpr (INT8) {
            const uint32_t* p = reinterpret_cast<const uint32_t*>(base) + hd * (kD * kD / 4) +
                                i * (kD / 4) + lane;
            uint32_t w;
            asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(w) : "l"(p));
            return codes4(w);
        } else {
            return ld_stream4(reinterpret_cast<const float*>(base) + hd * (kD * kD) + i * kD +
                              4 * lane);
        }
    }
    static __device__ __forceinline__ float4 coherent(const void* base, size_t hd, int i, int lane) {
        if constexpr (INT8) {
            const uint32_t* p = reinterpret_cast<const uint32_t*>(base) + hd * (kD * kD / 4) +
                                i * (kD / 4) + lane;
            return codes4(__ldcg(p));
        } else {
            return ldcg4(reinterpret_cast<const float*>(base) + hd * (kD * kD) + i * kD + 4 * lane);
        }
    }
};

// Symmetric INT8 codes of 4 values with a common scale, packed little-endian.
__device__ __forceinline__ uint32_t pack_codes4(float4 v, float s) {
    const uint32_t a = static_cast<uint32_t>(quant_code(v.x, s)) & 0xffu;
    const uint32_t b = static_cast<uint32_t>(quant_code(v.y, s)) & 0xffu;
    const uint32_t c = static_cast<uint32_t>(quant_code(v.z, s)) & 0xffu;
    const uint32_t d = static_cast<uint32_t>(quant_code(v.w, s)) & 0xffu;
    return a | (b << 8) | (c << 16) | (d << 24);
}

enum FoldMode : int { kFoldCommit = 0, kFoldRead = 1 };

constexpr int kFoldRows = 8;  // key rows folded per block

// Fold the first `n` log entries of state hd into its base, 8 key rows at a
// time (a warp holds 8 x 128 accumulators):
//     S[i][:] = exp(lb_i) dequant(B)[i][:] + sum_{l<n} exp(lb_i - Lam_l,i) K_l,i U_l[:]
// ("DeltaLog: Deferred Materialization of Recurrent States for Linear
// Attention Decoding", §3.2 eq. 7; eq. 6 when the log holds the current
// token, whose snapshot equals lb).  lb is the cumulative log-decay the log
// is folded at: per key row in lb_s (shared memory, per-key gate) or the
// scalar lb (scalar gate).
//   kFoldCommit: deferred -> S is the new FP32 base;  INT8 -> per key row
//     s_i = max_j |S_ij| / 127, codes rint(S / s_i) clamped to [-127, 127]
//     ("LeapQuant: Efficient Linear Attention with Accurate Recurrent State
//     Quantization", §3.2 eq. 4, App. B.3) -- written in place;
//   kFoldRead: S is written to out ([d_k][d_v]) and the pool is unchanged.
template <bool INT8, bool PER_KEY, int MODE>
__device__ __forceinline__ void fold_warp(const PoolView& pv, size_t hd, int n,
                                          const float* lb_s, float lb, float* out, int lane) {
    const size_t e0 = hd * static_cast<size_t>(pv.W);
#pragma unroll 1
    for (int i0 = 0; i0 < kD; i0 += kFoldRows) {
        float4 acc[kFoldRows];
        // decayed, dequantized base rows
#pragma unroll
        for (int r = 0; r < kFoldRows; ++r) {
            const int i = i0 + r;
            float e = expf(PER_KEY ? lb_s[i] : lb);
            if constexpr (INT8) e *= __ldcg(pv.scale + hd * kD + i);
            const float4 b = BaseRows<INT8>::coherent(pv.base, hd, i, lane);
            acc[r] = make_float4(e * b.x, e * b.y, e * b.z, e * b.w);
        }
        // + sum_l exp(lb - Lam_l) K_l U_l^T
#pragma unroll 1
        for (int l = 0; l < n; ++l) {
            const size_t eo = (e0 + l) * kD;
            const float4 ka = ldcg4(pv.klog + eo + i0);
            const float4 kb = ldcg4(pv.klog + eo + i0 + 4);
            const float4 u = ldcg4(pv.ulog + eo + 4 * lane);
            float a[kFoldRows] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
            if constexpr (PER_KEY) {
                const float4 la = ldcg4(pv.lamlog + eo + i0);
                const float4 lc = ldcg4(pv.lamlog + eo + i0 + 4);
                const float lm[kFoldRows] = {la.x, la.y, la.z, la.w, lc.x, lc.y, lc.z, lc.w};
#pragma unroll
                for (int r = 0; r < kFoldRows; ++r) a[r] *= expf(lb_s[i0 + r] - lm[r]);
            } else {
                const float g = expf(lb - __ldcg(pv.lamlog + e0 + l));
#pragma unroll
                for (int r = 0; r < kFoldRows; ++r) a[r] *= g;
            }
#pragma unroll
            for (int r = 0; r < kFoldRows; ++r) {
                acc[r].x = fmaf(a[r], u.x, acc[r].x);
                acc[r].y = fmaf(a[r], u.y, acc[r].y);
                acc[r].z = fmaf(a[r], u.z, acc[r].z);
                acc[r].w = fmaf(a[r], u.w, acc[r].w);
            }
        }
        // write the block
#pragma unroll
        for (int r = 0; r < kFoldRows; ++r) {
            const int i = i0 + r;
            if constexpr (MODE == kFoldRead) {
                st4(out + i * kD + 4 * lane, acc[r]);
            } else if constexpr (!INT8) {
                st4(reinterpret_cast<float*>(pv.base) + hd * (kD * kD) + i * kD + 4 * lane, acc[r]);
            } else {
                float m = fmaxf(fmaxf(fabsf(acc[r].x), fabsf(acc[r].y)),
                                fmaxf(fabsf(acc[r].z), fabsf(acc[r].w)));
                m = warp_max(m);
                const float s = __fdiv_rn(m, 127.0f);
                reinterpret_cast<uint32_t*>(pv.base)[hd * (kD * kD / 4) + i * (kD / 4) + lane] =
                    pack_codes4(acc[r], s);
                if (lane == 0) pv.scale[hd * kD + i] = s;
            }
        }
    }
}

}  // namespace ls
