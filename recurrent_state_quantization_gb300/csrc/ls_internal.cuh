// ls_internal.cuh -- private declarations of libls (pool layout, kernel
// arguments, launchers).  Shared only by the library's own translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include <utility>

struct ls_pool;  // the opaque handle of ls.h

namespace ls {

// The device that was current when the pool was created (its memory's device).
int pool_device(const ::ls_pool* p);

constexpr int kD = 128;         // d_k = d_v
constexpr int kThreads = 256;   // threads of every CTA (8 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kSplitEntries = 6;  // split replay: log entries per streamed chunk

// Device status word bits (mirror LS_DEV_* of ls.h).
constexpr int32_t kDevSlotRange = 1;
constexpr int32_t kDevTimeout = 2;
constexpr int32_t kDevBadState = 4;
constexpr int32_t kDevSlotDup = 8;

// Device pointers into one pool (caller-owned memory).  "hd" below is the
// state index slot * H + h.
//
// Base layouts:
//   eager FP32        S^T, [P*H][d_v][d_k]: value column j holds the 128 key
//                     rows contiguously (the eager kernel stages whole tiles
//                     in shared memory and reduces columns over 8 lanes);
//   deferred FP32     S,   [P*H][d_k][d_v]: key row i holds the 128 value
//                     columns contiguously (one warp owns a head, each lane
//                     4 value columns; a row is one 512-byte warp access and
//                     a key row's absmax is a warp reduction);
//   INT8              S in 4x4 column quads: byte (i, j) of a head sits at
//                     ((i/4) * 32 + j/4) * 16 + (j%4) * 4 + i%4, so a 32-bit
//                     word holds 4 key rows of one value column (one dp4a
//                     operand) and 32 lanes read 4 whole rows in one 512-byte
//                     access (lane l: columns 4l..4l+3).
struct PoolView {
    int32_t* status;       // [1] LS_DEV_* bits
    void* base;            // FP32 or INT8 base states (see above)
    float* scale;          // INT8: [P*H][d_k] key-row factors: per-row scales s,
                           //   or the smoothing factors c (column-scale format)
    float* colf;           // INT8 column-scale format: [P*H][d_v] value-column
                           //   scales b; nullptr for per-row scales
    float* lbar;           // log variants: [P*H][dl] cumulative log-decay
    int32_t* len;          // log variants: [P*H] live log length
    float* klog;           // [P*H][cap][d_k]  key factors k (bfloat16 when k16,
                           //   binary16 when rec16)
    float* ulog;           // [P*H][cap][d_v]  value factors u (binary16 when rec16)
    float* lamlog;         // [P*H][lam_stride] cumulative log-decay snapshots:
                           //   per-key gate [cap][d_k]; scalar gate [cap] padded to 4
    int32_t P, H, W, dl;
    int32_t R;             // INT8: compensator pairs at the head of each window (0: none)
    int32_t plain;         // 1: update pair (k, v), no delta-rule correction
    int32_t k16;           // 1: klog holds bfloat16
    int32_t rec16;         // 1: klog and ulog hold IEEE binary16 (INT8 FP16 records)
    int32_t cap;           // log entries per state: W + R
    int32_t lam_stride;    // floats per state in lamlog
    int32_t* foldq;        // INT8 without compensator pairs:
                           //   window-end queue [0] count, [2] done, [1] and
                           //   [3] unused, [4 ..] (state index, request row)
                           //   pairs (the tensor-core window-end kernel's work
                           //   list); nullptr otherwise
    int32_t fold_grid;     // CTAs of the window-end fold kernel (the SM count)
    int32_t* mark;         // LS_CHECK_SLOTS: [P] per-slot counts of the slot
                           //   check, zero between calls; nullptr otherwise
};

struct StepArgs {
    PoolView pv;
    const int32_t* slot_idx;
    int32_t batch;
    const float* q;
    const float* k;
    const float* v;
    const float* lam;
    const float* beta;
    float* y;
    float2* coef;     // split replay: [batch * H][cstride] (c_k, c_q) per log entry
    int32_t cstride;  // entries per row, a multiple of kSplitEntries
};

struct AuxArgs {
    PoolView pv;
    const int32_t* slots;  // [n]
    int32_t n;
    const float* state_in;  // load: [n][H][d_k][d_v]
    float* state_out;       // read: [n][H][d_k][d_v]
    int8_t* codes_out;      // read_int8: [n][H][d_k][d_v]
    float* scales_out;      // read_int8: [n][H][d_k]
    int32_t* len_out;       // read_log_meta: [n][H]
    float* lbar_out;        // read_log_meta: [n][H][dl]
};

// ---- shared-memory footprints (bytes) -------------------------------------
constexpr size_t kVecBytes = kD * sizeof(float);
__host__ __device__ constexpr size_t tile_bytes(bool int8) {
    return int8 ? size_t(kD) * kD : size_t(kD) * kD * 4;
}
constexpr size_t kMiscBytes = 128;
constexpr size_t kBarBytes = 64;
__host__ __device__ constexpr size_t eager_smem_bytes() {
    return tile_bytes(false) + 6 * kVecBytes + kMiscBytes + kBarBytes;
}
__host__ __device__ constexpr size_t transpose_smem_bytes() { return size_t(kD) * (kD + 1) * 4; }

// ---- launchers (each in its own translation unit) -------------------------
// Launch a step kernel with programmatic stream serialization allowed, so it
// may be scheduled while the previous kernel on the stream drains (the
// kernel itself waits for that kernel before touching memory).
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, size_t smem, cudaStream_t s,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t prepare_eager_step_kernels();
cudaError_t prepare_log_step_kernels();
cudaError_t prepare_fold_kernels();
cudaError_t prepare_aux_kernels();
cudaError_t prepare_window_fold_kernels();
cudaError_t prepare_int8_step_kernels();

cudaError_t launch_eager_step(const StepArgs& a, bool per_key, cudaStream_t s);
cudaError_t launch_log_step(const StepArgs& a, bool int8, bool per_key, cudaStream_t s);
cudaError_t launch_log_step_split(const StepArgs& a, bool int8, bool per_key, cudaStream_t s);
// INT8 pools with a window-end queue: the lean INT8 step kernel (fused or
// split replay), then the window-end fold.
cudaError_t launch_int8_step(const StepArgs& a, bool per_key, bool split, cudaStream_t s);
// INT8 pools with a window-end queue: decode the tokens the step kernel just
// queued, fold each state's log and requantize it (a no-op launch when the
// queue is empty).
cudaError_t launch_window_fold(const StepArgs& a, bool per_key, cudaStream_t s);
// deferred / INT8: fold the live log into the base (commit) or into a caller
// buffer (read) for n slots.
cudaError_t launch_fold(const AuxArgs& a, bool int8, bool per_key, bool commit, cudaStream_t s);
cudaError_t launch_eager_read(const AuxArgs& a, cudaStream_t s);
cudaError_t launch_load(const AuxArgs& a, bool int8, bool has_log, cudaStream_t s);
cudaError_t launch_reset(const AuxArgs& a, bool int8, bool has_log, cudaStream_t s);
cudaError_t launch_read_int8(const AuxArgs& a, cudaStream_t s);
cudaError_t launch_read_colf(const AuxArgs& a, cudaStream_t s);
cudaError_t launch_read_comp(const AuxArgs& a, cudaStream_t s);
cudaError_t launch_init_comp(const PoolView& pv, cudaStream_t s);
cudaError_t launch_read_log_meta(const AuxArgs& a, cudaStream_t s);
cudaError_t launch_slot_check(const PoolView& pv, const int32_t* slots, int32_t n, cudaStream_t s);

}  // namespace ls
