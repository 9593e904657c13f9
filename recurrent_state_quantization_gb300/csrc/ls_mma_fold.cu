// ls_mma_fold.cu -- INT8 window ends on the 5th-generation tensor cores
// (tcgen05, sm_103a).
//
// At a window end of an INT8 pool with per-row scales and no compensator
// pairs, the step kernel appends the closing token (the log then holds all W
// records) and queues the state.  This kernel, launched after every such
// step, folds each queued state and requantizes it:
//     S[i][j] = exp(lb_i) s_i Z_ij + sum_{l<W} exp(lb_i - Lam_l,i) K_l,i U_l,j
//     B_i = max_j |S_ij|,  s_i = B_i / 127,  Z_ij = rint(S_ij 127 / B_i)
// ("LeapQuant: Efficient Linear Attention with Accurate Recurrent State
// Quantization", §3.2 eq. 4 and App. B.3; "DeltaLog: Deferred Materialization
// of Recurrent States for Linear Attention Decoding", §3.2 eq. 6: the merge
// as base decay plus the decayed records), then resets lbar and the log.
//
// The rank-W part is a GEMM, D = U^T A with D[j][i] (value column j in
// tensor-memory lane j, key row i in column i), A[i][l] = exp(lb_i - Lam_l,i)
// K_l,i and U[j][l] = U_l,j: M = N = 128, K = W, 16 records per chunk.  Each
// FP32 operand is split into its TF32 rounding and the exact FP32 remainder,
// x = x_h + x_r, and D accumulates U_h A_h + U_h A_r + U_r A_h (three
// kind::tf32 MMAs per 8 records).  The dropped U_r A_r term and the TF32
// reading of the remainders leave about 2^-22 relative error per product,
// FP32-level accuracy, so the codes match an FP32 fold but for rounding ties.
//
// A kernel that allocates tensor memory runs one CTA per SM (measured: the
// occupancy calculator and the hardware both give 1, whatever the shared
// memory), so this kernel is persistent, one CTA of 512 threads per SM, and
// the step kernel carries no tcgen05 code at all.  The CTA holds four
// independent groups of 128 threads.  A group takes the next queued state;
// its records and codes were staged in shared memory by bulk copies while
// the group finished the previous state.  Each thread reads its row of the
// raw records, the group builds the split operands in place (K-major core
// matrices, see ls_umma.cuh), one thread issues the MMAs into the group's 128
// tensor-memory columns and commits them to the group's mbarrier, and the
// copies of the next state start as soon as the MMAs have read the operands.
// The epilogue runs on the CUDA cores: thread t of a group owns value column
// j = t (the tensor-memory lanes its warp may read) for all 128 key rows.
// The INT8 words of a state hold 4 key rows of one value column, so each
// thread reads and writes 32 whole words and a warp 128 contiguous bytes per
// access; a key row's absmax over a warp's 32 columns is one redux.sync, over
// the group's 4 warps a shared-memory max.
// S goes back to tensor memory between the absmax pass and the quantization
// pass, so no thread holds more than 32 of its 128 values.
//
// Queue protocol (pool memory, zeroed at creation): the step kernel appends
// state indices after atomically incrementing count; here groups take items
// by atomically incrementing next; the last CTA to finish resets count, next
// and done to zero for the next token.  With an empty queue every CTA returns
// at once.
#include <cuda_runtime.h>

#include "ls_device.cuh"
#include "ls_internal.cuh"
#include "ls_umma.cuh"
#include "ls_warp.cuh"

namespace ls {

namespace {

constexpr int kGroups = 4;
constexpr int kGroupThreads = 128;
constexpr int kFoldThreads = kGroups * kGroupThreads;
constexpr int kChunkRecords = 16;                            // records per MMA chunk
constexpr uint32_t kOperandBytes = kD * kChunkRecords * 4;   // one operand copy: 8 KiB
constexpr uint32_t kCodeBytes = kD * kD;                     // INT8 codes of one state

// Shared memory of one group.  The raw records of a chunk are staged by bulk
// copies inside the operand buffers (U in ops[1], K in ops[3], the per-key
// log-decay snapshots in ops[2]) and turned into the split operands in place
// once every thread holds its row in registers.
struct alignas(128) GroupSmem {
    unsigned char ops[4][kOperandBytes];  // U head, U remainder, A head, A remainder
    uint32_t codes[kCodeBytes / 4];       // old codes of the state being folded
    float vs[kD];                         // staged old scales s_i
    float vl[kD];                         // staged lbar (per-key gate)
    float es[kD];                         // exp(lb_i) s_i
    float red[4][kD];                     // per-warp absmax of each key row
    float fq[kD];                         // 127 / B_i
    float gl[kChunkRecords];              // scalar gate: exp(lb - Lam_l) of the chunk
    uint64_t ld_bar;                      // records (+ s, lbar) of a chunk
    uint64_t cw_bar;                      // codes
    uint64_t mma_bar;                     // MMA completion
    int32_t next_item;                    // queue position of the next state
    float next_lb;                        // scalar gate: lbar of the next state
};

constexpr size_t window_fold_smem_bytes() { return kGroups * sizeof(GroupSmem); }
static_assert(window_fold_smem_bytes() <= 232448, "the four groups fit one CTA's shared memory (227 KiB)");

// K-major core-matrix offset of records 4q..4q+3 of operand row `row`
// (8-row groups 512 B apart, 4-record groups 128 B apart).
__device__ __forceinline__ uint32_t operand_offset(int row, int q) {
    return static_cast<uint32_t>((row >> 3) * 512 + q * 128 + (row & 7) * 16);
}

// OR of pred over the nthreads threads of barrier id (a barrier itself).
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Stage records c0 .. c0 + nl - 1 of state hd (and, for the first chunk, its
// scales and per-key lbar) on ld_bar (one thread).
template <bool PER_KEY>
__device__ __forceinline__ void stage_records(const PoolView& pv, size_t hd, int c0, int nl, GroupSmem& gs) {
    const size_t eo = (hd * static_cast<size_t>(pv.cap) + c0) * kD;
    const uint32_t part = static_cast<uint32_t>(nl) * kVecBytes;
    const uint32_t kpart = static_cast<uint32_t>(nl) * kD * key_bytes(pv);
    const uint32_t upart = static_cast<uint32_t>(nl) * kD * val_bytes(pv);
    const size_t lb0 = hd * static_cast<size_t>(pv.lam_stride);
    const uint32_t lam_bytes = PER_KEY ? part : static_cast<uint32_t>((nl + 3) / 4 * 16);
    uint32_t bytes = upart + kpart + lam_bytes;
    if (c0 == 0) bytes += kVecBytes + (PER_KEY ? kVecBytes : 0);
    fence_proxy_async();  // the buffers were last used by generic loads and stores
    mbar_arrive_expect_tx(&gs.ld_bar, bytes);
    bulk_g2s(gs.ops[1], reinterpret_cast<const unsigned char*>(pv.ulog) + eo * val_bytes(pv), upart, &gs.ld_bar);
    bulk_g2s(gs.ops[3], reinterpret_cast<const unsigned char*>(pv.klog) + eo * key_bytes(pv), kpart, &gs.ld_bar);
    if constexpr (PER_KEY)
        bulk_g2s(gs.ops[2], pv.lamlog + lb0 + static_cast<size_t>(c0) * kD, part, &gs.ld_bar);
    else
        bulk_g2s(gs.ops[2], pv.lamlog + lb0 + c0, lam_bytes, &gs.ld_bar);
    if (c0 == 0) {
        bulk_g2s(gs.vs, pv.scale + hd * kD, kVecBytes, &gs.ld_bar);
        if constexpr (PER_KEY) bulk_g2s(gs.vl, pv.lbar + hd * kD, kVecBytes, &gs.ld_bar);
    }
}

// Stage the 16 KiB of codes of state hd on cw_bar (one thread).
__device__ __forceinline__ void stage_codes(const PoolView& pv, size_t hd, GroupSmem& gs) {
    const unsigned char* src = reinterpret_cast<const unsigned char*>(pv.base) + hd * kCodeBytes;
    fence_proxy_async();
    mbar_arrive_expect_tx(&gs.cw_bar, kCodeBytes);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        bulk_g2s(reinterpret_cast<unsigned char*>(gs.codes) + i * (kCodeBytes / 4), src + i * (kCodeBytes / 4),
                 kCodeBytes / 4, &gs.cw_bar);
}

// Three MMAs per 8 records of the staged chunk (one thread).
__device__ __forceinline__ void issue_chunk(const GroupSmem& gs, uint32_t tmem, int nl, bool accumulate) {
    const uint32_t a_hi = smem_u32(gs.ops[0]), a_lo = smem_u32(gs.ops[1]);
    const uint32_t b_hi = smem_u32(gs.ops[2]), b_lo = smem_u32(gs.ops[3]);
    const int ks = (nl + 7) >> 3;
    for (int s = 0; s < ks; ++s) {
        const uint32_t o = 256u * s;  // two 4-record core-matrix columns per MMA
        umma_tf32(tmem, umma_desc(a_hi + o, 128, 512), umma_desc(b_hi + o, 128, 512),
                  (accumulate || s > 0) ? 1u : 0u);
        umma_tf32(tmem, umma_desc(a_hi + o, 128, 512), umma_desc(b_lo + o, 128, 512), 1u);
        umma_tf32(tmem, umma_desc(a_lo + o, 128, 512), umma_desc(b_hi + o, 128, 512), 1u);
    }
}

// Per-group pipeline state: barrier phases and which copies / MMAs are in
// flight.
struct GroupPipe {
    uint32_t ld_ph = 0, cw_ph = 0, mma_ph = 0;
    bool ld_out = false, cw_out = false, mma_out = false;
};

// Wait (bounded) for one phase of bar; group-uniform result.  On a timeout
// the status is flagged and false returned.
__device__ __forceinline__ bool group_wait(const PoolView& pv, uint64_t* bar, uint32_t& phase, bool& out,
                                           int bar_id, int gt) {
    const bool ok = mbar_wait_bounded(bar, phase);
    if (named_barrier_or(bar_id, kGroupThreads, !ok)) {
        if (gt == 0) flag_status(pv.status, kDevTimeout);
        return false;
    }
    phase ^= 1u;
    out = false;
    return true;
}

// Fold and requantize state hd with the 128 threads of one group (gt = thread
// in the group, gw = its warp in the group).  On entry the first chunk of its
// records and its codes are staged or in flight.  Thread 0 takes the next
// queue item early; once the last MMA has read the operands it stages that
// state's first chunk, and once pass 1 has read the codes, its codes, so the
// copies overlap this state's epilogue.  Returns false after a timeout
// (flagged).
template <bool PER_KEY>
__device__ __forceinline__ bool fold_state(const PoolView& pv, size_t hd, float lb_scalar, GroupSmem& gs,
                                           GroupPipe& gp, uint32_t tmem, uint32_t tlane, int bar_id, int gt,
                                           int lane, int gw, int count) {
    const int n = pv.cap;  // W records (no compensator pairs on this path)
    int next_item = 0;
    long long next_hd = -1;
    float next_lb = 0.0f;
    if (gt == 0) {  // the next state, early: its index is needed once the MMAs are done
        next_item = atomicAdd(pv.foldq + 1, 1);
        if (next_item < count) {
            next_hd = __ldcg(pv.foldq + 4 + next_item);
            if constexpr (!PER_KEY) next_lb = __ldcg(pv.lbar + next_hd);
        }
    }
    float lb = lb_scalar;  // the cumulative log-decay the log is folded at (row gt)
#pragma unroll 1
    for (int c0 = 0; c0 < n; c0 += kChunkRecords) {
        const int nl = min(kChunkRecords, n - c0);
        if (!group_wait(pv, &gs.ld_bar, gp.ld_ph, gp.ld_out, bar_id, gt)) return false;
        if (c0 == 0) {
            if constexpr (PER_KEY) lb = gs.vl[gt];
            gs.es[gt] = expf(lb) * gs.vs[gt];
        }
        // row gt of both operands: U_l[j = gt] and A[i = gt][l] = exp(lb_i - Lam_l,i) K_l,i
        // (scalar gate: one factor per record, computed once for the group)
        const float* ru = reinterpret_cast<const float*>(gs.ops[1]);
        const float* rl = reinterpret_cast<const float*>(gs.ops[2]);
        float u[kChunkRecords], x[kChunkRecords];
        if (!PER_KEY && gt < kChunkRecords) gs.gl[gt] = gt < nl ? expf(lb - rl[gt]) : 0.0f;
#pragma unroll
        for (int l = 0; l < kChunkRecords; ++l) {
            u[l] = 0.0f;
            x[l] = 0.0f;
            if (l < nl) {
                u[l] = pv.rec16 ? __half2float(reinterpret_cast<const __half*>(gs.ops[1])[l * kD + gt])
                                : ru[l * kD + gt];
                x[l] = (pv.k16 || pv.rec16)
                           ? key16_to_float(reinterpret_cast<const unsigned short*>(gs.ops[3])[l * kD + gt],
                                            pv.k16 != 0)
                           : reinterpret_cast<const float*>(gs.ops[3])[l * kD + gt];
                if constexpr (PER_KEY) x[l] *= expf(lb - rl[l * kD + gt]);
            }
        }
        named_barrier(bar_id, kGroupThreads);  // every row is in registers: the buffers are free
        if constexpr (!PER_KEY) {
#pragma unroll
            for (int l = 0; l < kChunkRecords; ++l) x[l] *= gs.gl[l];
        }
#pragma unroll
        for (int qq = 0; qq < kChunkRecords / 4; ++qq) {
            const uint32_t off = operand_offset(gt, qq);
            float4 h = make_float4(tf32_rna(u[4 * qq]), tf32_rna(u[4 * qq + 1]), tf32_rna(u[4 * qq + 2]),
                                   tf32_rna(u[4 * qq + 3]));
            *reinterpret_cast<float4*>(gs.ops[0] + off) = h;
            *reinterpret_cast<float4*>(gs.ops[1] + off) =
                make_float4(u[4 * qq] - h.x, u[4 * qq + 1] - h.y, u[4 * qq + 2] - h.z, u[4 * qq + 3] - h.w);
            h = make_float4(tf32_rna(x[4 * qq]), tf32_rna(x[4 * qq + 1]), tf32_rna(x[4 * qq + 2]),
                            tf32_rna(x[4 * qq + 3]));
            *reinterpret_cast<float4*>(gs.ops[2] + off) = h;
            *reinterpret_cast<float4*>(gs.ops[3] + off) =
                make_float4(x[4 * qq] - h.x, x[4 * qq + 1] - h.y, x[4 * qq + 2] - h.z, x[4 * qq + 3] - h.w);
        }
        fence_proxy_async();  // the operand stores, before the tensor cores read them
        named_barrier(bar_id, kGroupThreads);
        if (gt == 0) {
            tc_fence_after();
            issue_chunk(gs, tmem, nl, c0 > 0);
            umma_commit(&gs.mma_bar);
            gp.mma_out = true;
        }
        if (!group_wait(pv, &gs.mma_bar, gp.mma_ph, gp.mma_out, bar_id, gt)) return false;
        // the operands are consumed: stage the next chunk, or the next state's first
        if (gt == 0) {
            if (c0 + kChunkRecords < n) {
                stage_records<PER_KEY>(pv, hd, c0 + kChunkRecords, min(kChunkRecords, n - c0 - kChunkRecords), gs);
                gp.ld_out = true;
            } else if (next_hd >= 0) {
                stage_records<PER_KEY>(pv, static_cast<size_t>(next_hd), 0, min(kChunkRecords, n), gs);
                gp.ld_out = true;
            }
        }
    }
    tc_fence_after();
    if (!group_wait(pv, &gs.cw_bar, gp.cw_ph, gp.cw_out, bar_id, gt)) return false;
    // pass 1: S = D + the decayed, dequantized old base, 32 key rows at a
    // time; each row's absmax over this warp's columns; S back to tensor memory
#pragma unroll
    for (int qr = 0; qr < 4; ++qr) {
        float d[32];
        tmem_ld32(tlane + 32u * qr, d);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const uint32_t w = gs.codes[(8 * qr + g) * kD + gt] ^ 0x80808080u;
            const float4 e4 = reinterpret_cast<const float4*>(gs.es)[8 * qr + g];
            const float2 z01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650)),
                                                      __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7651))),
                                          make_float2(-kCodeBias, -kCodeBias));
            const float2 z23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7652)),
                                                      __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7653))),
                                          make_float2(-kCodeBias, -kCodeBias));
            const float2 s01 = __ffma2_rn(z01, make_float2(e4.x, e4.y), make_float2(d[4 * g], d[4 * g + 1]));
            const float2 s23 = __ffma2_rn(z23, make_float2(e4.z, e4.w), make_float2(d[4 * g + 2], d[4 * g + 3]));
            d[4 * g + 0] = s01.x;
            d[4 * g + 1] = s01.y;
            d[4 * g + 2] = s23.x;
            d[4 * g + 3] = s23.y;
        }
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            const float4 m = make_float4(warp_absmax_redux(d[c]), warp_absmax_redux(d[c + 1]),
                                         warp_absmax_redux(d[c + 2]), warp_absmax_redux(d[c + 3]));
            if (lane == 0) reinterpret_cast<float4*>(gs.red[gw])[8 * qr + c / 4] = m;
        }
        tmem_st32(tlane + 32u * qr, d);
    }
    tc_fence_before();
    if (gt == 0) {
        gs.next_item = next_item;
        gs.next_lb = next_lb;
    }
    named_barrier(bar_id, kGroupThreads);  // row maxima complete, codes consumed
    if (gt == 0 && next_hd >= 0) {
        stage_codes(pv, static_cast<size_t>(next_hd), gs);
        gp.cw_out = true;
    }
    {
        const float B = fmaxf(fmaxf(gs.red[0][gt], gs.red[1][gt]), fmaxf(gs.red[2][gt], gs.red[3][gt]));
        float sc, f;
        row_quant_params(B, sc, f);
        pv.scale[hd * kD + gt] = sc;
        gs.fq[gt] = f;
    }
    named_barrier(bar_id, kGroupThreads);
    tc_fence_after();
    // pass 2: codes rint(S 127 / B_i), four key rows per word, one warp
    // writing 128 contiguous bytes per store
    uint32_t* const words = reinterpret_cast<uint32_t*>(pv.base) + hd * (kCodeBytes / 4) + gt;
#pragma unroll
    for (int qr = 0; qr < 4; ++qr) {
        float d[32];
        tmem_ld32(tlane + 32u * qr, d);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const float4 f4 = reinterpret_cast<const float4*>(gs.fq)[8 * qr + g];
            const float2 a = code_words2(make_float2(d[4 * g], d[4 * g + 1]), make_float2(f4.x, f4.y));
            const float2 b = code_words2(make_float2(d[4 * g + 2], d[4 * g + 3]), make_float2(f4.z, f4.w));
            words[(8 * qr + g) * kD] = pack_low_bytes(a.x, a.y, b.x, b.y);
        }
    }
    tc_fence_before();  // these reads, before the group's next MMAs (after a barrier)
    // a new window starts at this boundary
    if constexpr (PER_KEY) {
        pv.lbar[hd * kD + gt] = 0.0f;
    } else if (gt == 0) {
        pv.lbar[hd] = 0.0f;
    }
    if (gt == 0) pv.len[hd] = pv.R;
    return true;
}

template <bool PER_KEY>
__global__ void __launch_bounds__(kFoldThreads, 1) window_fold_kernel(const PoolView pv) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t tmem_base;
    __shared__ int32_t count_s;
    pdl_enter();
    int32_t* const q = pv.foldq;
    const int tid = threadIdx.x;
    if (tid == 0) count_s = __ldcg(q);
    __syncthreads();
    const int count = count_s;
    if (count <= 0) return;  // no window closed on this token
    const int warp = tid >> 5, lane = tid & 31;
    const int g = warp >> 2, gt = tid & (kGroupThreads - 1), gw = warp & 3;
    GroupSmem& gs = reinterpret_cast<GroupSmem*>(smem)[g];
    const int bar_id = 1 + g;
    GroupPipe gp;
    if (gt == 0) {
        mbar_init(&gs.ld_bar, 1);
        mbar_init(&gs.cw_bar, 1);
        mbar_init(&gs.mma_bar, 1);
        mbar_fence_init();
        // the group's first state
        const int item = atomicAdd(q + 1, 1);
        gs.next_item = item;
        if (item < count) {
            const size_t hd = static_cast<size_t>(__ldcg(q + 4 + item));
            if constexpr (!PER_KEY) gs.next_lb = __ldcg(pv.lbar + hd);
            stage_records<PER_KEY>(pv, hd, 0, min(kChunkRecords, pv.cap), gs);
            stage_codes(pv, hd, gs);
            gp.ld_out = gp.cw_out = true;
        }
    }
    if (warp == 0) tmem_alloc512(&tmem_base);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base + 128u * g;                           // the group's columns
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * gw) << 16);  // the warp's lanes
    int item = gs.next_item;
    float lb = gs.next_lb;
#pragma unroll 1
    while (item < count) {
        const size_t hd = static_cast<size_t>(__ldcg(q + 4 + item));
        if (!fold_state<PER_KEY>(pv, hd, lb, gs, gp, tmem, tlane, bar_id, gt, lane, gw, count)) {
            // after a timeout: let this group's copies and MMAs land before exit
            if (gt == 0) {
                if (gp.ld_out) mbar_wait_bounded(&gs.ld_bar, gp.ld_ph);
                if (gp.cw_out) mbar_wait_bounded(&gs.cw_bar, gp.cw_ph);
                if (gp.mma_out) mbar_wait_bounded(&gs.mma_bar, gp.mma_ph);
            }
            break;
        }
        item = gs.next_item;
        lb = gs.next_lb;
    }
    tc_fence_before();
    __syncthreads();  // every group is done with tensor memory and the queue
    if (warp == 0) tmem_dealloc512(tmem_base);
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(q + 2, 1) == static_cast<int>(gridDim.x) - 1) {
            q[0] = 0;
            q[1] = 0;
            q[2] = 0;
        }
    }
}

}  // namespace

cudaError_t prepare_window_fold_kernels() {
    const int bytes = static_cast<int>(window_fold_smem_bytes());
    cudaError_t e = cudaFuncSetAttribute(window_fold_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(window_fold_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_window_fold(const PoolView& pv, bool per_key, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pv.fold_grid > 0 ? pv.fold_grid : 1));
    cfg.blockDim = dim3(kFoldThreads);
    cfg.dynamicSmemBytes = window_fold_smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return per_key ? cudaLaunchKernelEx(&cfg, window_fold_kernel<true>, pv)
                   : cudaLaunchKernelEx(&cfg, window_fold_kernel<false>, pv);
}

}  // namespace ls
