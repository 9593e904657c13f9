/*
 * ls.h -- C ABI of libls: the per-token decode step of delta-rule linear
 * attention over a pool of recurrent states, on NVIDIA GB300 (sm_103a).
 *
 * Per head, with S a d_k x d_v state (d_k = d_v = 128), one token computes
 *     S_t = (I - beta k k^T) D_t S_{t-1} + beta k v^T,     y_t = S_t^T q_t,
 * with D_t = alpha_t I (Gated DeltaNet, scalar gate) or D_t = Diag(alpha_t)
 * (KDA, per-key gate).  Expanded as in "LeapQuant: Efficient Linear Attention
 * with Accurate Recurrent State Quantization", App. A (GDN / KDA rows):
 *     u = beta (v - S_{t-1}^T (alpha . k)),  S_t = D_t S_{t-1} + k u^T.
 * The gate is passed as a log-decay lambda = log(alpha) <= 0, as in
 * "DeltaLog: Deferred Materialization of Recurrent States for Linear
 * Attention Decoding", §2.1 eq. 2-3.
 *
 * Three storage variants sit behind the same calls:
 *   LS_EAGER_FP32     dense FP32 state, read, updated and written every token.
 *   LS_DEFERRED_FP32  dense FP32 base + a bounded log of per-token factors
 *                     (k, u, cumulative log-decay); every read is served
 *                     exactly from base + log, and the log is folded into the
 *                     base every `window` tokens (DeltaLog §3.1 Algorithm 1,
 *                     eq. 4-7, merge interval M = window).
 *   LS_WINDOW_INT8    INT8 base with one FP32 scale per key row, held fixed
 *                     for a window of `window` tokens while the tokens'
 *                     updates are buffered in FP32; outputs come from the
 *                     dequantized base plus the buffer; the state is
 *                     re-quantized only at the window's end (LeapQuant §3.2
 *                     eq. 3-4; readout App. B.2 eq. 9; window = 1 is the
 *                     per-step quantization of eq. 2).
 *
 * Conventions of every call
 *   - Device memory (the pool, inputs, outputs) is owned by the caller; the
 *     library never allocates device memory.  Host-side, a pool handle is a
 *     small malloc'ed struct.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on it, except ls_pool_create's layout checks and
 *     ls_pool_status, which synchronizes it.  Pointers must stay valid until
 *     the stream reaches the call.
 *   - Every call returns an int status: LS_OK (0) or a negative LS_ERR_*.
 *     Argument errors are detected on the host before anything is launched
 *     (nothing is changed).  Errors only the device can see (a slot index out
 *     of range, a bounded wait that gave up) are recorded in the pool's
 *     status word, read by ls_pool_status; the affected head is skipped and
 *     its output row is filled with NaN.
 *   - No C++ exception crosses the ABI.  Calls on one pool must not overlap
 *     on different streams.
 *   - Inputs and outputs are FP32, row-major, contiguous.
 */
#ifndef LS_H_
#define LS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LS_ABI_VERSION 5

/* status codes */
#define LS_OK 0
#define LS_ERR_INVALID (-1) /* null pointer, bad enum, bad descriptor       */
#define LS_ERR_ALIGN (-2)   /* a pointer is not aligned as documented       */
#define LS_ERR_SLOT (-3)    /* slot list longer than the pool can hold      */
#define LS_ERR_CUDA (-4)    /* a CUDA runtime call or kernel launch failed  */
#define LS_ERR_SIZE (-5)    /* unsupported size, or a buffer too small      */

/* bits of the device status word (ls_pool_status) */
#define LS_DEV_SLOT_RANGE 1 /* a slot index outside [0, num_slots) was skipped */
#define LS_DEV_TIMEOUT 2    /* a bounded wait on an asynchronous copy gave up  */
#define LS_DEV_BAD_STATE 4  /* a state's log length was out of range (its pool
                               memory was overwritten); the state was skipped */
#define LS_DEV_SLOT_DUP 8   /* a slot list held one slot more than once
                               (pools created with LS_CHECK_SLOTS)            */

typedef struct ls_pool ls_pool; /* opaque host handle */

typedef enum {
    LS_EAGER_FP32 = 0,
    LS_DEFERRED_FP32 = 1,
    LS_WINDOW_INT8 = 2
} ls_variant;

typedef enum {
    LS_GATE_SCALAR = 0, /* Gated DeltaNet: log_decay is [batch, H]      */
    LS_GATE_PER_KEY = 1 /* KDA: log_decay is [batch, H, d_k]             */
} ls_gate;

/* Largest `window` (W for LS_WINDOW_INT8, M for LS_DEFERRED_FP32). */
#define LS_MAX_WINDOW 256

/*
 * ls_pool_desc.flags.  LS_INT8_COLUMN_SCALES (LS_WINDOW_INT8 only): store the
 * window-boundary state in the smoothed per-value-column format of
 * "LeapQuant: Efficient Linear Attention with Accurate Recurrent State
 * Quantization", §3.4 eq. 7 and App. B.3: each key row i is divided by its
 * smoothing factor c_i = max(sqrt(mean_j |S_ij|), 2^-20), and the result is
 * quantized with one symmetric INT8 scale b_j = B_j / 127 per value column
 * (B_j the column's absmax, codes rint(R_ij * (127 / B_j))), so that
 * S_ij ~ c_i Z_ij b_j; reads use eq. 10 (B Z^T C Gamma x / 127).  Without
 * the flag, one scale s_i = B_i / 127 per key row: S_ij ~ s_i Z_ij.
 */
#define LS_INT8_COLUMN_SCALES 1u

/*
 * ls_pool_desc.flags, bits 8..11: r Compensator Tokens (LS_WINDOW_INT8 only,
 * 0 <= r <= LS_MAX_COMPENSATORS), "LeapQuant: Efficient Linear Attention with
 * Accurate Recurrent State Quantization", §3.3 eq. 5-6: at every window
 * boundary (window end, ls_window_commit, ls_pool_load) r rank-one pairs
 * (k~, u~) are fitted to the state by power iteration and kept as FP32 log
 * records with log-decay snapshot 0 at the head of the next window; only
 * the residual S - K~ U~^T is quantized.  The fit: sequential deflation, per
 * pair three steps v <- R^T R v / ||R^T R v|| from all-ones / sqrt(d_v),
 * then k~ = R v, u~ = v.  A state's log then holds r + (real tokens)
 * entries, and its window ends on its W-th real token.
 */
#define LS_MAX_COMPENSATORS 8

/*
 * ls_pool_desc.flags: LS_PLAIN_UPDATE (LS_EAGER_FP32 / LS_DEFERRED_FP32):
 * the update pair is the raw (k_t, v_t) with no delta-rule correction,
 * S_t = D_t S_{t-1} + k_t v_t^T, y_t = S_t^T q_t: the linear attention,
 * RetNet, GLA and RWKV6 rows of "DeltaLog: Deferred Materialization of
 * Recurrent States for Linear Attention Decoding", Table 1 (RWKV6 = the
 * per-key gate).  beta is passed as usual but its values are not used.
 */
#define LS_PLAIN_UPDATE (1u << 12)

/*
 * ls_pool_desc.flags: LS_LOG_BF16_K (LS_DEFERRED_FP32 / LS_WINDOW_INT8,
 * without compensator pairs): the key-side factors of the log are stored
 * as bfloat16 (round to nearest even), the value-side factors and decay
 * snapshots stay FP32 ("DeltaLog: Deferred Materialization of Recurrent
 * States for Linear Attention Decoding", §3.4).  Reads of later tokens use
 * the stored factor; the token's own output, and a merge that folds it,
 * use k.  A log entry shrinks by 2 d_k bytes.
 */
#define LS_LOG_BF16_K (1u << 13)

/*
 * ls_pool_desc.flags: LS_INT8_FP16_RECORDS (LS_WINDOW_INT8 only, not with
 * LS_LOG_BF16_K): the window's buffered records -- the keys k and the
 * corrected values u -- and the compensator pairs are stored in IEEE
 * binary16, rounded to nearest even; the decay snapshots stay FP32 ("LeapQuant:
 * Efficient Linear Attention with Accurate Recurrent State Quantization", §4.1:
 * FP16 Compensator Tokens; §4.3: the FP16 update buffer of a window).  The
 * token's own output uses k and u; later reads, the window end and the state
 * use the stored records.  A scalar-gate record takes 516 bytes instead of
 * 1028.  Values beyond the binary16 range become infinite (not checked).
 */
#define LS_INT8_FP16_RECORDS (1u << 14)

/*
 * ls_pool_desc.flags: LS_CHECK_SLOTS (every variant): a checking mode for
 * callers.  Every call that changes states -- the decode steps,
 * ls_pool_load, ls_pool_reset_slots, ls_window_commit of a log variant --
 * first checks on the device that its slot list names no slot twice: one
 * extra launch of one CTA, which counts each slot in a per-slot array of the
 * pool, tests the counts and clears them.  A repeated slot sets
 * LS_DEV_SLOT_DUP in the status word (ls_pool_status).  The call itself
 * still runs, so the states of a repeated slot are then undefined, as
 * without the flag.  The pool holds 4 more bytes per slot.
 */
#define LS_CHECK_SLOTS (1u << 15)
#define LS_INT8_COMPENSATORS(r) ((uint32_t)(r) << 8)

typedef struct {
    int32_t num_slots; /* P >= 1: states (requests) the pool holds            */
    int32_t num_heads; /* H >= 1                                                */
    int32_t d_k;       /* must be 128                                          */
    int32_t d_v;       /* must be 128                                          */
    int32_t variant;   /* ls_variant                                           */
    int32_t gate;      /* ls_gate                                              */
    int32_t window;    /* W (INT8) or M (deferred), 1..LS_MAX_WINDOW; ignored
                          (may be 0) for LS_EAGER_FP32                          */
    uint32_t flags;    /* 0; for LS_WINDOW_INT8 also LS_INT8_COLUMN_SCALES,
                          LS_INT8_COMPENSATORS(r) and LS_INT8_FP16_RECORDS; for
                          the FP32 variants also LS_PLAIN_UPDATE; LS_LOG_BF16_K
                          for the log variants; LS_CHECK_SLOTS for any */
} ls_pool_desc;

/* Human-readable name of a status code.  Never NULL. */
const char *ls_error_string(int status);

/* LS_ABI_VERSION of the library. */
int ls_abi_version(void);

/*
 * Device bytes a pool with this descriptor needs.  The layout behind them is
 * private; it holds, per (slot, head): the base state (FP32 or INT8 + FP32
 * key-row scales), and for the deferred/INT8 variants the cumulative
 * log-decay, the live log length and `window` log entries (K: d_k floats,
 * U: d_v floats, log-decay snapshot: 1 or d_k floats) -- DeltaLog §3.1's
 * physical state; plus a status word.
 * Errors: LS_ERR_INVALID (bad descriptor or NULL), LS_ERR_SIZE (d != 128,
 * window out of range, or the size overflows).
 */
int ls_pool_required_bytes(const ls_pool_desc *desc, size_t *bytes);

/*
 * Bind a pool to caller-owned device memory `dev_mem` (>= required bytes,
 * 256-byte aligned) and zero it on `stream`: every state starts at S = 0 with
 * an empty log / a window boundary (the zero state is exact in INT8); with
 * compensator pairs the log holds the zero state's pairs (k~ = 0, u~ =
 * 1 / sqrt(d_v)), as after ls_pool_reset_slots.
 * `*out` receives the host handle.  The memory stays owned by the caller and
 * must outlive the handle.
 * Errors: LS_ERR_INVALID, LS_ERR_SIZE (bytes too small, bad descriptor),
 * LS_ERR_ALIGN (dev_mem), LS_ERR_CUDA.
 */
int ls_pool_create(const ls_pool_desc *desc, void *dev_mem, size_t bytes,
                   void *stream, ls_pool **out);

/* Free the host handle (not the device memory).  NULL is accepted. */
int ls_pool_destroy(ls_pool *pool);

/*
 * Overwrite the states of `n` slots with d_state, a device array
 * [n, H, d_k, d_v] (FP32, logical layout S[i][j], i = key row).  The slots'
 * logs are emptied (a window boundary).  For LS_WINDOW_INT8 the state is
 * quantized here (per key row, as at a window end).  This is how a prefill
 * output enters a fresh slot (DeltaLog §4, state-slot lifecycle).
 * d_slots: device int32 [n], distinct.  n = 0 is a no-op.
 * Errors: LS_ERR_INVALID, LS_ERR_ALIGN (d_state not 16-byte aligned),
 * LS_ERR_SLOT (n > num_slots), LS_ERR_CUDA.  Out-of-range slots are skipped
 * and flagged in the status word.
 */
int ls_pool_load(ls_pool *pool, const int32_t *d_slots, int32_t n,
                 const float *d_state, void *stream);

/* Zero the states of `n` slots and empty their logs (slot reuse). */
int ls_pool_reset_slots(ls_pool *pool, const int32_t *d_slots, int32_t n,
                        void *stream);

/*
 * One decode token for `batch` requests.  Row b of every input belongs to
 * pool slot d_slot_idx[b] (device int32 [batch], distinct, in [0, P)).
 *   q, k      [batch, H, d_k]   (16-byte aligned)
 *   v         [batch, H, d_v]   (16-byte aligned)
 *   log_decay [batch, H] (LS_GATE_SCALAR) or [batch, H, d_k] (LS_GATE_PER_KEY,
 *             16-byte aligned); values <= 0 (alpha = exp(log_decay))
 *   beta      [batch, H]
 *   y         [batch, H, d_v]   output (16-byte aligned), the post-update
 *             readout S_t^T q_t of the logical state.
 * Eager: S is read, updated and written.  Deferred / INT8: the base is read,
 * the token's factors (k, u, cumulative log-decay) are appended to the log;
 * on the window-th token since the slot's last boundary the log is folded
 * into the base (FP32 for deferred; re-quantized per key row for INT8, after
 * y was read from the unquantized state).  Different slots may be at
 * different positions of their windows.  An INT8 pool with per-row scales
 * and no compensator pairs queues its closing states in its own memory and
 * folds them in a second kernel on the tensor cores, launched on the same
 * stream by this call (every call; it ends at once when no window closed);
 * the other formats fold inside the step kernel.
 * batch = 0 is a no-op.  Errors: LS_ERR_INVALID, LS_ERR_ALIGN, LS_ERR_SLOT
 * (batch > num_slots), LS_ERR_SIZE (batch * H >= 2^31), LS_ERR_CUDA.
 */
int ls_decode_step(ls_pool *pool, const int32_t *d_slot_idx, int32_t batch,
                   const float *q, const float *k, const float *v,
                   const float *log_decay, const float *beta, float *y,
                   void *stream);

/*
 * Split replay (DeltaLog §5.3, the split-replay ablation): the decode token
 * of ls_decode_step for the deferred and INT8 variants as two kernels.  The
 * first writes, per (request, head), the replay coefficients of every live
 * log entry l,
 *   c_k[l] = K_l . (exp(lp - Lam_l) . k),  c_q[l] = K_l . (exp(lp - Lam_l) . q)
 * (lp the cumulative log-decay after this token), into the caller's device
 * scratch d_scratch; the second streams the base and the U side of the log
 * and applies those coefficients.  Same arguments, results and pool state as
 * ls_decode_step, bit for bit.  d_scratch: >= ls_split_scratch_bytes bytes,
 * 16-byte aligned, owned by the caller, contents on entry ignored; the call
 * reads and writes it in stream order, so calls that share one scratch
 * buffer must be ordered on one stream.  Errors: as ls_decode_step,
 * LS_ERR_INVALID (eager pool, null scratch), LS_ERR_ALIGN, LS_ERR_SIZE
 * (scratch smaller than required).
 */
int ls_decode_step_split(ls_pool *pool, const int32_t *d_slot_idx,
                         int32_t batch, const float *q, const float *k,
                         const float *v, const float *log_decay,
                         const float *beta, float *y, void *d_scratch,
                         size_t scratch_bytes, void *stream);

/*
 * Scratch bytes ls_decode_step_split needs for `batch` requests:
 * batch * H * ceil(capacity / 6) * 6 * 8, the capacity being the window /
 * merge interval plus the compensator pairs.  LS_ERR_INVALID for an eager
 * pool.
 */
int ls_split_scratch_bytes(const ls_pool *pool, int32_t batch, size_t *bytes);

/*
 * ls_decode_step_split without caller scratch.  No counterpart in the
 * papers: an allocation-free form of the split-replay step for callers that
 * cannot provide device scratch.  The coefficients go to one fixed device
 * array of LS_SPLIT_STATIC_SCRATCH_BYTES per device (library-owned, placed
 * by the CUDA runtime when the library's module loads); its address is
 * looked up once per device.  The pool's device (the one current at
 * ls_pool_create) must be the current device: otherwise the call returns
 * LS_ERR_INVALID and launches nothing.  The call allocates nothing.  No part of the array has to start at zero.
 * Overlapping calls race: every call on a device uses the same array, so
 * two calls whose kernels may run at the same time (different streams,
 * different host threads) corrupt each other's coefficients; order them on
 * one stream.  Arguments, results and errors as ls_decode_step_split, and
 * LS_ERR_SIZE when ls_split_scratch_bytes(pool, batch) exceeds
 * LS_SPLIT_STATIC_SCRATCH_BYTES (nothing is launched then).
 */
#define LS_SPLIT_STATIC_SCRATCH_BYTES (16u << 20)
int ls_decode_step_split_static(ls_pool *pool, const int32_t *d_slot_idx,
                                int32_t batch, const float *q, const float *k,
                                const float *v, const float *log_decay,
                                const float *beta, float *y, void *stream);

/*
 * Device bytes of the staging buffer ls_decode_step_host needs for `batch`.
 */
int ls_step_staging_bytes(const ls_pool *pool, int32_t batch, size_t *bytes);

/*
 * ls_decode_step with HOST inputs and output: copies h_slot_idx, h_q, h_k,
 * h_v, h_log_decay, h_beta (same shapes as above, host memory, ideally
 * pinned) into the caller's device staging buffer d_staging (>= the bytes
 * of ls_step_staging_bytes, 256-byte aligned) with cudaMemcpyAsync, runs the
 * step, and copies y back into h_y, all on `stream`.  The host buffers must
 * stay valid until the stream reaches the call (synchronize before reading
 * h_y).  Errors: as ls_decode_step, LS_ERR_SIZE (staging too small).
 */
int ls_decode_step_host(ls_pool *pool, const int32_t *h_slot_idx,
                        int32_t batch, const float *h_q, const float *h_k,
                        const float *h_v, const float *h_log_decay,
                        const float *h_beta, float *h_y, void *d_staging,
                        size_t staging_bytes, void *stream);

/*
 * Close the current window / merge cycle of `n` slots now, without a new
 * token: deferred -> fold the log into the FP32 base (DeltaLog eq. 6 without
 * the a_t b_t^T term); INT8 -> fold and re-quantize; eager -> no-op.  A slot
 * whose log is empty is left unchanged.  The logical state does not change
 * (up to INT8 rounding).  Errors as ls_pool_load.
 */
int ls_window_commit(ls_pool *pool, const int32_t *d_slots, int32_t n,
                     void *stream);

/*
 * Write the logical state of `n` slots into d_state_out [n, H, d_k, d_v]
 * (FP32, logical layout S[i][j]) without changing the pool: DeltaLog §3.2
 * eq. 7 for deferred, LeapQuant §3.2 eq. 4 (from the dequantized base) for
 * INT8.  Errors as ls_pool_load.
 */
int ls_pool_read(const ls_pool *pool, const int32_t *d_slots, int32_t n,
                 float *d_state_out, void *stream);

/*
 * LS_WINDOW_INT8 only: the current base of `n` slots as codes
 * d_codes [n, H, d_k, d_v] (int8, logical layout, 16-byte aligned) and the
 * key-row factors d_scales [n, H, d_k] (FP32): the per-row scales s_i, so
 * dequant(S)[i][j] = s_i * codes[i][j]; with LS_INT8_COLUMN_SCALES the
 * smoothing factors c_i (see ls_pool_read_int8_col_scales).  Errors as
 * ls_pool_load, and LS_ERR_INVALID for the other variants.
 */
int ls_pool_read_int8(const ls_pool *pool, const int32_t *d_slots, int32_t n,
                      int8_t *d_codes, float *d_scales, void *stream);

/*
 * LS_WINDOW_INT8 with LS_INT8_COLUMN_SCALES only: the per-value-column
 * scales b_j of `n` slots into d_col_scales [n, H, d_v] (FP32), so that
 * dequant(S)[i][j] = c_i * codes[i][j] * b_j (LeapQuant App. B.3).  Errors
 * as ls_pool_load, and LS_ERR_INVALID for other pools.
 */
int ls_pool_read_int8_col_scales(const ls_pool *pool, const int32_t *d_slots,
                                 int32_t n, float *d_col_scales, void *stream);

/*
 * LS_WINDOW_INT8 with LS_INT8_COMPENSATORS(r), r >= 1, only: the current
 * window's compensator pairs of `n` slots into d_k_out [n, H, r, d_k] and
 * d_u_out [n, H, r, d_v] (FP32).  Errors as ls_pool_load, and
 * LS_ERR_INVALID for other pools.
 */
int ls_pool_read_compensators(const ls_pool *pool, const int32_t *d_slots,
                              int32_t n, float *d_k_out, float *d_u_out,
                              void *stream);

/*
 * Deferred / INT8 only: the live log length of every (slot, head) into
 * d_len [n, H] (int32) and, when d_lbar is not NULL, the cumulative
 * log-decay into d_lbar [n, H, 1] (scalar gate) or [n, H, d_k] (per-key).
 */
int ls_pool_read_log_meta(const ls_pool *pool, const int32_t *d_slots,
                          int32_t n, int32_t *d_len, float *d_lbar,
                          void *stream);

/*
 * Synchronize `stream`, return the pool's device status word in
 * *device_status (0 or LS_DEV_* bits) and clear it.
 */
int ls_pool_status(ls_pool *pool, void *stream, int32_t *device_status);

#ifdef __cplusplus
}
#endif

#endif /* LS_H_ */
