// ls_mma_fold.cu -- INT8 window ends on the 5th-generation tensor cores
// (tcgen05, sm_103a).
//
// A token that closes an INT8 state's window (per-row scales or the
// smoothed column-scale format, no compensator pairs) is not decoded by the
// step kernel: it queues (state, request row), and this kernel, launched
// right after every such step, decodes it in one pass over the state
// (LeapQuant §3.2 eq. 3-4 with App. A; DeltaLog §3.2 eq. 6, the merge that
// includes the current update):
//     lp   = lbar + lambda                          (cumulative log-decay)
//     S    = exp(lp_i) s_i Z_ij + sum_{l<n} exp(lp_i - Lam_l,i) K_l,i U_l,j
//          = D_t S_{t-1}, the decayed logical state (n = W - 1 stored records)
//     r    = S^T k,  y0 = S^T q,  u = beta (v - r),  y = y0 + (k.q) u
//     S   += k u^T   (with bfloat16 keys or binary16 records: the factors as a
//                     record would store them; y uses k and u themselves)
//     B_i  = max_j |S_ij|,  s_i = B_i / 127,  Z_ij = rint(S_ij 127 / B_i)
// (App. B.3), then lbar = 0 and the log is emptied.  y is read from the
// unquantized state.  The column-scale format (LeapQuant §3.4 eq. 7, App.
// B.3) dequantizes the old base as c_i Z_ij b_j and quantizes the new state
// as c_i = max(sqrt(mean_j |S_ij|), 2^-20), R = S / c (row-wise), b_j =
// max_i |R_ij| / 127, Z_ij = rint(R_ij 127 / max_i |R_ij|).  The codes and the records of a closing state are read
// once, here.
//
// The rank-n part is a GEMM, D = U^T A with D[j][i] (value column j in
// tensor-memory lane j, key row i in column i), A[i][l] = exp(lp_i - Lam_l,i)
// K_l,i and U[j][l] = U_l,j: M = N = 128, K = n, 16 records per chunk.  Each
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
// its header (the token's k, q, v, the state's scales, and for the per-key
// gate lambda and lbar), codes and first records were staged in shared
// memory by bulk copies while the group finished the previous state.  Each
// thread reads its row of the raw records, the group builds the split
// operands in place (K-major core matrices, see ls_umma.cuh), one thread
// issues the MMAs into the group's 128 tensor-memory columns and commits them
// to the group's mbarrier, and the copies of the next state start as soon as
// the MMAs have read the operands (records) and pass 2 is done with the
// codes (codes, header); lane 0 of each of the group's four warps issues a
// part of them, so that no warp arrives late at the next group barrier.  The
// epilogue runs on the CUDA cores: thread t of a group
// owns value column j = t (the tensor-memory lanes its warp may read) for
// all 128 key rows, so r_j, y0_j and u_j are thread-local sums.  The INT8
// words of a state hold 4 key rows of one value column, so each thread reads
// and writes 32 whole words and a warp 128 contiguous bytes per access; a
// key row's absmax over a warp's 32 columns is one redux.sync, over the
// group's 4 warps a shared-memory max (column scales: a row's sum of |S| by a
// 31-shuffle reduce-scatter over the warp; a column's absmax is
// thread-local).  Pass 1 forms S (32 key rows at a time) and the readouts
// and puts S back in tensor memory; pass 2 adds k u^T, takes the row
// statistics and puts S back again; (column scales: pass 3 puts R = S / c
// back and takes the column's absmax;) the last pass writes the codes, so
// no thread holds more than 32 of its 128 values.
//
// Queue protocol (pool memory, zeroed at creation): the step kernel appends
// (state, row) pairs after atomically incrementing count; here the items are
// dealt round-robin over the groups of the grid (group g of CTA b takes
// items 4 b + g, 4 b + g + 4 grid, ...), so that each group knows its next
// item's position without an atomic and loads its entry one state ahead;
// the last CTA to finish resets count and done to zero for the next token.
// With an empty queue every CTA returns at once.
//
// The record format (FP32, bfloat16 keys, binary16 records) is a template
// parameter, like the step kernels', so that the operand build reads each
// record element without a branch on the format.
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
    float hk[kD];                         // header of the state: its closing token's
    float hq[kD];                         //   k, q, v, its key-row scales s, and for
    float hv[kD];                         //   the per-key gate lambda and lbar
    float hs[kD];
    float hlam[kD];
    float hlb[kD];
    float hb[kD];                         // column-scale format: the old scales b_j
    float kk[kD];                         // the key of the state update, as a record
                                          //   stores it (the header is restaged
                                          //   after pass 2)
    float es[kD];                         // exp(lp_i) s_i
    float red[4][kD];                     // per-warp absmax of each key row
    float fq[kD];                         // 127 / B_i (per-row scales) or the row
                                          //   factors g_i = 1 / c_i (column scales)
    float gl[kChunkRecords];              // scalar gate: exp(lp - Lam_l) of the chunk
    float kqp[4];                         // per-warp partial sums of k.q
    uint64_t rec_bar;                     // records of a chunk
    uint64_t st_bar;                      // codes + header of a state
    uint64_t mma_bar;                     // MMA completion
    int32_t next_item;                    // queue position of the next state
    int32_t next_hd, next_row;            // the next state and its request row
    float next_lb, next_lam, next_beta;   // its lbar, lambda (scalar gate) and beta
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

// Queue item `item`: (state index, request row).
__device__ __forceinline__ int2 queue_item(const PoolView& pv, int item) {
    return __ldcg(reinterpret_cast<const int2*>(pv.foldq + 4) + item);
}

// Part p (0..3) of the staging of records c0 .. c0 + nl - 1 of state hd,
// issued by lane 0 of the group's warp p on rec_bar (arrival count 4): U,
// K, the log-decay snapshots, or (p = 3) an arrival alone.
template <bool PER_KEY, int REC>
__device__ __forceinline__ void stage_records_part(const PoolView& pv, size_t hd, int c0, int nl, GroupSmem& gs,
                                                   int p) {
    constexpr uint32_t kb = rec_key_bytes(REC), vb = rec_val_bytes(REC);
    const size_t eo = (hd * static_cast<size_t>(pv.cap) + c0) * kD;
    const size_t lb0 = hd * static_cast<size_t>(pv.lam_stride);
    fence_proxy_async();  // the buffers were last used by generic loads and stores
    if (p == 0) {
        const uint32_t upart = static_cast<uint32_t>(nl) * kD * vb;
        mbar_arrive_expect_tx(&gs.rec_bar, upart);
        bulk_g2s(gs.ops[1], reinterpret_cast<const unsigned char*>(pv.ulog) + eo * vb, upart, &gs.rec_bar);
    } else if (p == 1) {
        const uint32_t kpart = static_cast<uint32_t>(nl) * kD * kb;
        mbar_arrive_expect_tx(&gs.rec_bar, kpart);
        bulk_g2s(gs.ops[3], reinterpret_cast<const unsigned char*>(pv.klog) + eo * kb, kpart, &gs.rec_bar);
    } else if (p == 2) {
        if constexpr (PER_KEY) {
            const uint32_t part = static_cast<uint32_t>(nl) * kVecBytes;
            mbar_arrive_expect_tx(&gs.rec_bar, part);
            bulk_g2s(gs.ops[2], pv.lamlog + lb0 + static_cast<size_t>(c0) * kD, part, &gs.rec_bar);
        } else {
            const uint32_t lam_bytes = static_cast<uint32_t>((nl + 3) / 4 * 16);
            mbar_arrive_expect_tx(&gs.rec_bar, lam_bytes);
            bulk_g2s(gs.ops[2], pv.lamlog + lb0 + c0, lam_bytes, &gs.rec_bar);
        }
    } else {
        mbar_arrive_expect_tx(&gs.rec_bar, 0);
    }
}

// Part p (0..3) of the staging of state hd, issued by lane 0 of the group's
// warp p on st_bar (arrival count 4): code quarter p and a share of the
// header (k, q | v, s | lambda, lbar for the per-key gate | the old column
// scales), so that no warp of the group issues all the copies.
template <bool PER_KEY, bool COLS>
__device__ __forceinline__ void stage_state_part(const StepArgs& a, size_t hd, int row, GroupSmem& gs, int p) {
    const PoolView& pv = a.pv;
    const unsigned char* src = reinterpret_cast<const unsigned char*>(pv.base) + hd * kCodeBytes;
    const size_t ro = static_cast<size_t>(row) * kD;
    uint32_t bytes = kCodeBytes / 4;
    if (p == 0 || p == 1) bytes += 2 * kVecBytes;
    if (p == 2 && PER_KEY) bytes += 2 * kVecBytes;
    if (p == 3 && COLS) bytes += kVecBytes;
    fence_proxy_async();
    mbar_arrive_expect_tx(&gs.st_bar, bytes);
    bulk_g2s(reinterpret_cast<unsigned char*>(gs.codes) + p * (kCodeBytes / 4), src + p * (kCodeBytes / 4),
             kCodeBytes / 4, &gs.st_bar);
    if (p == 0) {
        bulk_g2s(gs.hk, a.k + ro, kVecBytes, &gs.st_bar);
        bulk_g2s(gs.hq, a.q + ro, kVecBytes, &gs.st_bar);
    } else if (p == 1) {
        bulk_g2s(gs.hv, a.v + ro, kVecBytes, &gs.st_bar);
        bulk_g2s(gs.hs, pv.scale + hd * kD, kVecBytes, &gs.st_bar);
    } else if (p == 2) {
        if constexpr (PER_KEY) {
            bulk_g2s(gs.hlam, a.lam + ro, kVecBytes, &gs.st_bar);
            bulk_g2s(gs.hlb, pv.lbar + hd * kD, kVecBytes, &gs.st_bar);
        }
    } else {
        if constexpr (COLS) bulk_g2s(gs.hb, pv.colf + hd * kD, kVecBytes, &gs.st_bar);
    }
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
    uint32_t rec_ph = 0, st_ph = 0, mma_ph = 0;
    bool rec_out = false, st_out = false, mma_out = false;
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

// The decayed, dequantized codes of key rows 32 qr .. 32 qr + 31 of value
// column gt added to d (the rank-n fold of those rows); bj is the column's
// scale (column-scale format) or 1.
template <bool COLS>
__device__ __forceinline__ void add_base_rows(const GroupSmem& gs, int qr, int gt, float bj, float (&d)[32]) {
    const float2 b2 = make_float2(bj, bj);
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
        const float2 s01 = __ffma2_rn(COLS ? __fmul2_rn(z01, b2) : z01, make_float2(e4.x, e4.y),
                                      make_float2(d[4 * g], d[4 * g + 1]));
        const float2 s23 = __ffma2_rn(COLS ? __fmul2_rn(z23, b2) : z23, make_float2(e4.z, e4.w),
                                      make_float2(d[4 * g + 2], d[4 * g + 3]));
        d[4 * g + 0] = s01.x;
        d[4 * g + 1] = s01.y;
        d[4 * g + 2] = s23.x;
        d[4 * g + 3] = s23.y;
    }
}

// Sum over the warp's 32 lanes of each of 32 per-lane values |v[r]| (one
// per key row), by recursive halving: 31 shuffles.  Lane l returns the sum
// for row l.
__device__ __forceinline__ float warp_abs_sum32_scatter(float (&v)[32], int lane) {
#pragma unroll
    for (int b = 4, h = 16; b >= 0; --b, h >>= 1) {
        const bool upper = (lane >> b) & 1;
#pragma unroll
        for (int r = 0; r < h; ++r) {
            const float send = upper ? v[r] : v[r + h];
            const float keep = upper ? v[r + h] : v[r];
            const float got = __shfl_xor_sync(0xffffffffu, send, 1 << b);
            v[r] = h == 16 ? fabsf(keep) + fabsf(got) : keep + got;
        }
    }
    return v[0];
}

// A key factor as a log record of format REC stores it: bfloat16, binary16
// or FP32, widened back to FP32.
template <int REC>
__device__ __forceinline__ float stored_key(float k) {
    if constexpr (REC == kRecBF16K) return __bfloat162float(__float2bfloat16_rn(k));
    if constexpr (REC == kRecFP16) return __half2float(__float2half_rn(k));
    return k;
}

// d[c] += k_i u for the 32 key rows i = 32 qr + c (the closing token's
// rank-one update of value column gt).
__device__ __forceinline__ void add_token_rows(const GroupSmem& gs, int qr, float u, float (&d)[32]) {
    const float2 uu = make_float2(u, u);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const float4 k4 = reinterpret_cast<const float4*>(gs.kk)[8 * qr + g];
        const float2 a = __ffma2_rn(make_float2(k4.x, k4.y), uu, make_float2(d[4 * g], d[4 * g + 1]));
        const float2 b = __ffma2_rn(make_float2(k4.z, k4.w), uu, make_float2(d[4 * g + 2], d[4 * g + 3]));
        d[4 * g + 0] = a.x;
        d[4 * g + 1] = a.y;
        d[4 * g + 2] = b.x;
        d[4 * g + 3] = b.y;
    }
}

// Decode the closing token of state hd (request row `row`), fold and
// requantize the state with the 128 threads of one group (gt = thread in the
// group, gw = its warp in the group).  On entry its header and codes, and its
// first records, are staged or in flight.  Thread 0 knows the group's next
// item (its queue entry was loaded during the previous state) and publishes
// it once every thread has read this state's; once the last MMA has read the
// operands the four warps stage that state's first records, and after pass 2
// (the codes and the header are consumed) its codes and header, so the copies
// overlap this state's epilogue.  Returns false after a timeout (flagged).
template <bool PER_KEY, bool COLS, int REC>
__device__ __forceinline__ bool fold_state(const StepArgs& a, size_t hd, int row, float lb_scalar,
                                           float lam_scalar, float beta, GroupSmem& gs, GroupPipe& gp,
                                           uint32_t tmem, uint32_t tlane, int bar_id, int gt, int lane, int gw,
                                           int count, int item, int stride, int2& ahead) {
    const PoolView& pv = a.pv;
    const int n = pv.cap - 1;  // stored records; the closing token itself is never stored
    const int next_item = item + stride;
    long long next_hd = -1;
    int next_row = 0;
    float next_lb = 0.0f, next_lam = 0.0f, next_beta = 0.0f;
    int2 after = make_int2(-1, 0);
    if (gt == 0 && next_item < count) {
        // the next state's queue entry was loaded during the previous state;
        // its scalars are needed after pass 2, the entry after it next time
        next_hd = ahead.x;
        next_row = ahead.y;
        if constexpr (!PER_KEY) {
            next_lb = __ldcg(pv.lbar + next_hd);
            next_lam = __ldg(a.lam + next_row);
        }
        next_beta = __ldg(a.beta + next_row);
        if (next_item + stride < count) after = queue_item(pv, next_item + stride);
    }
    // header and codes: lp of key row gt, exp(lp) s, the token's k.q
    if (!group_wait(pv, &gs.st_bar, gp.st_ph, gp.st_out, bar_id, gt)) return false;
    if (gt == 0) {  // every thread has read this state's entry: publish the next one's
        gs.next_item = next_item;
        gs.next_hd = static_cast<int32_t>(next_hd);
        gs.next_row = next_row;
    }
    const float lp = PER_KEY ? gs.hlb[gt] + gs.hlam[gt] : lb_scalar + lam_scalar;
    gs.es[gt] = expf(lp) * gs.hs[gt];
    // the key of the state update is the one a record would store (bfloat16
    // keys, binary16 records); the token's own output uses k itself
    gs.kk[gt] = stored_key<REC>(gs.hk[gt]);
    const float vj = gs.hv[gt];
    const float bj = COLS ? gs.hb[gt] : 1.0f;  // the old scale of this thread's value column
    {
        const float kq_part = warp_sum(gs.hk[gt] * gs.hq[gt]);
        if (lane == 0) gs.kqp[gw] = kq_part;
    }
#pragma unroll 1
    for (int c0 = 0; c0 < n; c0 += kChunkRecords) {
        const int nl = min(kChunkRecords, n - c0);
        if (!group_wait(pv, &gs.rec_bar, gp.rec_ph, gp.rec_out, bar_id, gt)) return false;
        // row gt of both operands: U_l[j = gt] and A[i = gt][l] = exp(lp_i - Lam_l,i) K_l,i
        // (scalar gate: one factor per record, computed once for the group)
        const float* ru = reinterpret_cast<const float*>(gs.ops[1]);
        const float* rl = reinterpret_cast<const float*>(gs.ops[2]);
        float u[kChunkRecords], x[kChunkRecords];
        if (!PER_KEY && gt < kChunkRecords) gs.gl[gt] = gt < nl ? expf(lp - rl[gt]) : 0.0f;
#pragma unroll
        for (int l = 0; l < kChunkRecords; ++l) {
            u[l] = 0.0f;
            x[l] = 0.0f;
            if (l < nl) {
                if constexpr (REC == kRecFP16)
                    u[l] = __half2float(reinterpret_cast<const __half*>(gs.ops[1])[l * kD + gt]);
                else
                    u[l] = ru[l * kD + gt];
                if constexpr (REC == kRecFP32)
                    x[l] = reinterpret_cast<const float*>(gs.ops[3])[l * kD + gt];
                else
                    x[l] = key16_to_float(reinterpret_cast<const unsigned short*>(gs.ops[3])[l * kD + gt],
                                          REC == kRecBF16K);
                if constexpr (PER_KEY) x[l] *= expf(lp - rl[l * kD + gt]);
            }
        }
        named_barrier(bar_id, kGroupThreads);  // every row is in registers: the buffers are free
        // the MMAs read the records of (nl + 7) / 8 k-steps of 8: only those are split and stored
        const bool half = nl <= kChunkRecords / 2;
        if constexpr (!PER_KEY) {
#pragma unroll
            for (int l = 0; l < kChunkRecords; ++l)
                if (!half || l < kChunkRecords / 2) x[l] *= gs.gl[l];
        }
#pragma unroll
        for (int qq = 0; qq < kChunkRecords / 4; ++qq) {
            if (half && qq >= kChunkRecords / 8) break;
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
        // the operands are consumed: stage the next chunk, or the next state's
        // first, a part per warp
        if (lane == 0) {
            if (c0 + kChunkRecords < n) {
                stage_records_part<PER_KEY, REC>(pv, hd, c0 + kChunkRecords, min(kChunkRecords, n - c0 - kChunkRecords),
                                            gs, gw);
                gp.rec_out = true;
            } else if (gs.next_hd >= 0) {
                stage_records_part<PER_KEY, REC>(pv, static_cast<size_t>(gs.next_hd), 0, min(kChunkRecords, n), gs, gw);
                gp.rec_out = true;
            }
        }
    }
    tc_fence_after();
    if (n == 0) named_barrier(bar_id, kGroupThreads);  // es, kk, k.q complete (with records,
                                                       // their barriers ordered these)
    // pass 1: S = D + the decayed, dequantized old base, 32 key rows at a
    // time; r = S^T k and y0 = S^T q of this thread's column; S back to
    // tensor memory
    float2 r2 = make_float2(0.f, 0.f), y2 = r2;
#pragma unroll
    for (int qr = 0; qr < 4; ++qr) {
        float d[32];
        if (n > 0) {
            tmem_ld32(tlane + 32u * qr, d);
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) d[c] = 0.0f;
        }
        add_base_rows<COLS>(gs, qr, gt, bj, d);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const float4 k4 = reinterpret_cast<const float4*>(gs.hk)[8 * qr + g];  // k itself
            const float4 q4 = reinterpret_cast<const float4*>(gs.hq)[8 * qr + g];
            r2 = __ffma2_rn(make_float2(d[4 * g], d[4 * g + 1]), make_float2(k4.x, k4.y), r2);
            r2 = __ffma2_rn(make_float2(d[4 * g + 2], d[4 * g + 3]), make_float2(k4.z, k4.w), r2);
            y2 = __ffma2_rn(make_float2(d[4 * g], d[4 * g + 1]), make_float2(q4.x, q4.y), y2);
            y2 = __ffma2_rn(make_float2(d[4 * g + 2], d[4 * g + 3]), make_float2(q4.z, q4.w), y2);
        }
        tmem_st32(tlane + 32u * qr, d);
    }
    const float kq = (gs.kqp[0] + gs.kqp[1]) + (gs.kqp[2] + gs.kqp[3]);
    // the closing token's correction and output (y from the unquantized state)
    const float r = r2.x + r2.y, y0 = y2.x + y2.y;
    const float u_out = beta * (vj - r);
    a.y[static_cast<size_t>(row) * kD + gt] = fmaf(kq, u_out, y0);
    const float uj = REC == kRecFP16 ? __half2float(__float2half_rn(u_out)) : u_out;  // as a record stores it
    // pass 2: S + k u^T back to tensor memory; per key row over this warp's
    // columns, the absmax (per-row scales) or the sum of |S| (column scales)
#pragma unroll
    for (int qr = 0; qr < 4; ++qr) {
        float d[32];
        tmem_ld32(tlane + 32u * qr, d);
        add_token_rows(gs, qr, uj, d);
        tmem_st32(tlane + 32u * qr, d);
        if constexpr (COLS) {
            gs.red[gw][32 * qr + lane] = warp_abs_sum32_scatter(d, lane);
        } else {
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                const float4 m = make_float4(warp_absmax_redux(d[c]), warp_absmax_redux(d[c + 1]),
                                             warp_absmax_redux(d[c + 2]), warp_absmax_redux(d[c + 3]));
                if (lane == 0) reinterpret_cast<float4*>(gs.red[gw])[8 * qr + c / 4] = m;
            }
        }
    }
    tc_fence_before();
    if (gt == 0) {
        gs.next_lb = next_lb;
        gs.next_lam = next_lam;
        gs.next_beta = next_beta;
        ahead = after;
    }
    named_barrier(bar_id, kGroupThreads);  // row statistics complete; codes and header consumed
    if (lane == 0 && gs.next_hd >= 0) {
        stage_state_part<PER_KEY, COLS>(a, static_cast<size_t>(gs.next_hd), gs.next_row, gs, gw);
        gp.st_out = true;
    }
    if constexpr (COLS) {
        // smoothing factor c_i = max(sqrt(mean_j |S_ij|), 2^-20) and g_i = 1 / c_i
        // (LeapQuant §3.4 eq. 7; the floor's value is a reading of the page)
        float c = sqrtf(((gs.red[0][gt] + gs.red[1][gt]) + (gs.red[2][gt] + gs.red[3][gt])) * (1.0f / kD));
        if (!(c >= kSmoothFloor)) c = kSmoothFloor;
        pv.scale[hd * kD + gt] = c;
        gs.fq[gt] = __fdiv_rn(1.0f, c);
    } else {
        const float B = fmaxf(fmaxf(gs.red[0][gt], gs.red[1][gt]), fmaxf(gs.red[2][gt], gs.red[3][gt]));
        float sc, f;
        row_quant_params(B, sc, f);
        pv.scale[hd * kD + gt] = sc;
        gs.fq[gt] = f;
    }
    named_barrier(bar_id, kGroupThreads);
    tc_fence_after();
    float fj = 0.0f;  // column-scale format: 127 / B_j of this thread's column
    if constexpr (COLS) {
        // pass 3: R = S g_i back to tensor memory, this column's absmax B_j
        float B = 0.0f;
#pragma unroll
        for (int qr = 0; qr < 4; ++qr) {
            float d[32];
            tmem_ld32(tlane + 32u * qr, d);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const float4 g4 = reinterpret_cast<const float4*>(gs.fq)[8 * qr + g];
                const float2 a2 = __fmul2_rn(make_float2(d[4 * g], d[4 * g + 1]), make_float2(g4.x, g4.y));
                const float2 b2 = __fmul2_rn(make_float2(d[4 * g + 2], d[4 * g + 3]), make_float2(g4.z, g4.w));
                d[4 * g] = a2.x;
                d[4 * g + 1] = a2.y;
                d[4 * g + 2] = b2.x;
                d[4 * g + 3] = b2.y;
                B = fmaxf(B, fmaxf(fmaxf(fabsf(a2.x), fabsf(a2.y)), fmaxf(fabsf(b2.x), fabsf(b2.y))));
            }
            tmem_st32(tlane + 32u * qr, d);
        }
        float bcol;
        row_quant_params(B, bcol, fj);  // b_j = B_j / 127, f_j = 127 / B_j (App. B.3)
        pv.colf[hd * kD + gt] = bcol;
    }
    // last pass: codes rint(S 127 / B_i), or rint(R_ij 127 / B_j), four key rows
    // per word, one warp writing 128 contiguous bytes per store
    uint32_t* const words = reinterpret_cast<uint32_t*>(pv.base) + hd * (kCodeBytes / 4) + gt;
#pragma unroll
    for (int qr = 0; qr < 4; ++qr) {
        float d[32];
        tmem_ld32(tlane + 32u * qr, d);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            float2 a2, b2;
            if constexpr (COLS) {
                a2 = code_words(make_float2(d[4 * g], d[4 * g + 1]), fj);
                b2 = code_words(make_float2(d[4 * g + 2], d[4 * g + 3]), fj);
            } else {
                const float4 f4 = reinterpret_cast<const float4*>(gs.fq)[8 * qr + g];
                a2 = code_words2(make_float2(d[4 * g], d[4 * g + 1]), make_float2(f4.x, f4.y));
                b2 = code_words2(make_float2(d[4 * g + 2], d[4 * g + 3]), make_float2(f4.z, f4.w));
            }
            words[(8 * qr + g) * kD] = pack_low_bytes(a2.x, a2.y, b2.x, b2.y);
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

template <bool PER_KEY, bool COLS, int REC>
__global__ void __launch_bounds__(kFoldThreads, 1) window_fold_kernel(const StepArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t tmem_base;
    __shared__ int32_t count_s;
    pdl_enter();
    const PoolView& pv = a.pv;
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
    const int n = pv.cap - 1;
    GroupPipe gp;
    // queue items are dealt round-robin: group gid takes gid, gid + stride, ...
    const int stride = static_cast<int>(gridDim.x) * kGroups;
    int2 ahead = make_int2(-1, 0);  // thread 0: the queue entry of the group's next item
    if (gt == 0) {
        mbar_init(&gs.rec_bar, 4);  // one arrival per warp of the group
        mbar_init(&gs.st_bar, 4);  // one arrival per warp of the group
        mbar_init(&gs.mma_bar, 1);
        mbar_fence_init();
        // the group's first state
        const int item = static_cast<int>(blockIdx.x) * kGroups + g;
        gs.next_item = item;
        if (item + stride < count) ahead = queue_item(pv, item + stride);
        if (item < count) {
            const int2 it = queue_item(pv, item);
            gs.next_hd = it.x;
            gs.next_row = it.y;
            if constexpr (!PER_KEY) {
                gs.next_lb = __ldcg(pv.lbar + it.x);
                gs.next_lam = __ldg(a.lam + it.y);
            }
            gs.next_beta = __ldg(a.beta + it.y);
        }
    }
    if (warp == 0) tmem_alloc512(&tmem_base);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (lane == 0 && gs.next_item < count) {  // the group's first state, a part per warp
        stage_state_part<PER_KEY, COLS>(a, static_cast<size_t>(gs.next_hd), gs.next_row, gs, gw);
        gp.st_out = true;
        if (n > 0) {
            stage_records_part<PER_KEY, REC>(pv, static_cast<size_t>(gs.next_hd), 0, min(kChunkRecords, n), gs, gw);
            gp.rec_out = true;
        }
    }
    const uint32_t tmem = tmem_base + 128u * g;                           // the group's columns
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * gw) << 16);  // the warp's lanes
    int item = gs.next_item;
#pragma unroll 1
    while (item < count) {
        const size_t hd = static_cast<size_t>(gs.next_hd);
        const int row = gs.next_row;
        const float lb = gs.next_lb, lam = gs.next_lam, beta = gs.next_beta;
        if (!fold_state<PER_KEY, COLS, REC>(a, hd, row, lb, lam, beta, gs, gp, tmem, tlane, bar_id, gt, lane, gw,
                                       count, item, stride, ahead)) {
            // after a timeout: let this group's copies and MMAs land before exit
            if (gt == 0) {
                if (gp.rec_out) mbar_wait_bounded(&gs.rec_bar, gp.rec_ph);
                if (gp.st_out) mbar_wait_bounded(&gs.st_bar, gp.st_ph);
                if (gp.mma_out) mbar_wait_bounded(&gs.mma_bar, gp.mma_ph);
            }
            break;
        }
        item = gs.next_item;
    }
    tc_fence_before();
    __syncthreads();  // every group is done with tensor memory and the queue
    if (warp == 0) tmem_dealloc512(tmem_base);
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(q + 2, 1) == static_cast<int>(gridDim.x) - 1) {
            q[0] = 0;
            q[2] = 0;
        }
    }
}

template <bool PER_KEY, bool COLS>
cudaError_t prepare_format(int bytes) {
    const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(window_fold_kernel<PER_KEY, COLS, kRecFP32>, attr, bytes)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(window_fold_kernel<PER_KEY, COLS, kRecBF16K>, attr, bytes)) != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(window_fold_kernel<PER_KEY, COLS, kRecFP16>, attr, bytes);
}

template <bool PER_KEY, bool COLS>
cudaError_t launch_format(const cudaLaunchConfig_t& cfg, const StepArgs& a) {
    if (a.pv.k16) return cudaLaunchKernelEx(&cfg, window_fold_kernel<PER_KEY, COLS, kRecBF16K>, a);
    if (a.pv.rec16) return cudaLaunchKernelEx(&cfg, window_fold_kernel<PER_KEY, COLS, kRecFP16>, a);
    return cudaLaunchKernelEx(&cfg, window_fold_kernel<PER_KEY, COLS, kRecFP32>, a);
}

}  // namespace

cudaError_t prepare_window_fold_kernels() {
    const int bytes = static_cast<int>(window_fold_smem_bytes());
    cudaError_t e;
    if ((e = prepare_format<false, false>(bytes)) != cudaSuccess) return e;
    if ((e = prepare_format<true, false>(bytes)) != cudaSuccess) return e;
    if ((e = prepare_format<false, true>(bytes)) != cudaSuccess) return e;
    return prepare_format<true, true>(bytes);
}

cudaError_t launch_window_fold(const StepArgs& a, bool per_key, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.pv.fold_grid > 0 ? a.pv.fold_grid : 1));
    cfg.blockDim = dim3(kFoldThreads);
    cfg.dynamicSmemBytes = window_fold_smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.pv.colf != nullptr) return per_key ? launch_format<true, true>(cfg, a) : launch_format<false, true>(cfg, a);
    return per_key ? launch_format<true, false>(cfg, a) : launch_format<false, false>(cfg, a);
}

}  // namespace ls
