// ls_api.cu -- the C ABI of libls (declared in include/ls.h): argument
// validation, the private pool layout, and kernel dispatch.  No call
// allocates device memory; the only host allocation is the pool handle.
#include <cstdint>
#include <cstring>
#include <new>

#include <cuda_runtime.h>

#include "../../include/ls.h"
#include "ls_internal.cuh"

struct ls_pool {
    ls_pool_desc desc;
    unsigned char* mem;
    size_t bytes;
    ls::PoolView view;
    int num_sms;
    int device;  // current device at ls_pool_create: the device of dev_mem
};

namespace {

using ls::kD;

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool is_log_variant(int32_t v) { return v == LS_DEFERRED_FP32 || v == LS_WINDOW_INT8; }

struct Layout {
    size_t status, base, scale, colf, lbar, len, klog, ulog, lamlog, foldq, mark, total;
};

// INT8 pools without compensator pairs (per-row or column scales) close
// their windows on the tensor cores, in a kernel of its own after the step.
bool int8_mma_fold(const ls_pool_desc* d) {
    return d->variant == LS_WINDOW_INT8 && ((d->flags >> 8) & 15u) == 0;
}

// Checks a descriptor; fills the layout when it is valid.
int make_layout(const ls_pool_desc* d, Layout* L) {
    if (d == nullptr || L == nullptr) return LS_ERR_INVALID;
    if (d->variant < LS_EAGER_FP32 || d->variant > LS_WINDOW_INT8) return LS_ERR_INVALID;
    const uint32_t int8_flags = LS_INT8_COLUMN_SCALES | LS_INT8_COMPENSATORS(15);
    if ((d->flags & ~(int8_flags | LS_PLAIN_UPDATE | LS_LOG_BF16_K | LS_INT8_FP16_RECORDS |
                      LS_CHECK_SLOTS)) != 0)
        return LS_ERR_INVALID;
    if ((d->flags & LS_INT8_FP16_RECORDS) &&
        (d->variant != LS_WINDOW_INT8 || (d->flags & LS_LOG_BF16_K)))
        return LS_ERR_INVALID;
    if ((d->flags & LS_LOG_BF16_K) && (!is_log_variant(d->variant) || ((d->flags >> 8) & 15u) != 0))
        return LS_ERR_INVALID;
    const uint32_t ncomp = (d->flags >> 8) & 15u;
    if ((d->flags & int8_flags) && d->variant != LS_WINDOW_INT8) return LS_ERR_INVALID;
    if ((d->flags & LS_PLAIN_UPDATE) && d->variant == LS_WINDOW_INT8) return LS_ERR_INVALID;
    if (ncomp > LS_MAX_COMPENSATORS) return LS_ERR_INVALID;
    if (d->gate != LS_GATE_SCALAR && d->gate != LS_GATE_PER_KEY) return LS_ERR_INVALID;
    if (d->num_slots < 1 || d->num_heads < 1) return LS_ERR_INVALID;
    if (d->d_k != kD || d->d_v != kD) return LS_ERR_SIZE;
    const bool log = is_log_variant(d->variant);
    if (log && (d->window < 1 || d->window > LS_MAX_WINDOW)) return LS_ERR_SIZE;
    const uint64_t nh = static_cast<uint64_t>(d->num_slots) * static_cast<uint64_t>(d->num_heads);
    if (nh > 0x7fffffffull) return LS_ERR_SIZE;  // grid rows (batch * H) fit int32
    // log capacity: the window's records plus the compensator pairs
    const uint64_t W = log ? static_cast<uint64_t>(d->window) + ((d->flags >> 8) & 15u) : 0;
    const uint64_t dl = d->gate == LS_GATE_PER_KEY ? kD : 1;
    const bool int8 = d->variant == LS_WINDOW_INT8;
    size_t off = 0;
    L->status = off;
    off = align_up(off + 256);  // status word
    L->base = off;
    off = align_up(off + nh * kD * kD * (int8 ? 1 : 4));
    L->scale = off;
    off = align_up(off + (int8 ? nh * kD * 4 : 0));
    L->colf = off;  // per-value-column scales (LS_INT8_COLUMN_SCALES)
    off = align_up(off + ((d->flags & LS_INT8_COLUMN_SCALES) ? nh * kD * 4 : 0));
    L->lbar = off;
    off = align_up(off + (log ? nh * dl * 4 : 0));
    L->len = off;
    off = align_up(off + (log ? nh * 4 : 0));
    const bool rec16 = (d->flags & LS_INT8_FP16_RECORDS) != 0;
    L->klog = off;
    off = align_up(off + nh * W * kD * (((d->flags & LS_LOG_BF16_K) || rec16) ? 2 : 4));
    L->ulog = off;
    off = align_up(off + nh * W * kD * (rec16 ? 2 : 4));
    L->lamlog = off;
    // scalar gate: one snapshot per entry, per-state stride padded to a
    // multiple of 4 floats so every state's snapshots start 16-byte aligned
    off = align_up(off + nh * (dl == 1 ? (W + 3) / 4 * 4 : W * dl) * 4);
    // window-end queue of the tensor-core fold (INT8 without compensator pairs)
    L->foldq = off;
    off = align_up(off + (int8_mma_fold(d) ? 16 + nh * 8 : 0));
    // per-slot counts of the duplicate-slot check
    L->mark = off;
    off = align_up(off + ((d->flags & LS_CHECK_SLOTS) ? static_cast<size_t>(d->num_slots) * 4 : 0));
    L->total = off;
    return LS_OK;
}

ls::PoolView make_view(const ls_pool_desc& d, const Layout& L, unsigned char* m) {
    const bool log = is_log_variant(d.variant);
    ls::PoolView v{};
    v.status = reinterpret_cast<int32_t*>(m + L.status);
    v.base = m + L.base;
    v.scale = d.variant == LS_WINDOW_INT8 ? reinterpret_cast<float*>(m + L.scale) : nullptr;
    v.colf = (d.flags & LS_INT8_COLUMN_SCALES) ? reinterpret_cast<float*>(m + L.colf) : nullptr;
    v.lbar = log ? reinterpret_cast<float*>(m + L.lbar) : nullptr;
    v.len = log ? reinterpret_cast<int32_t*>(m + L.len) : nullptr;
    v.klog = log ? reinterpret_cast<float*>(m + L.klog) : nullptr;
    v.ulog = log ? reinterpret_cast<float*>(m + L.ulog) : nullptr;
    v.lamlog = log ? reinterpret_cast<float*>(m + L.lamlog) : nullptr;
    v.P = d.num_slots;
    v.H = d.num_heads;
    v.W = log ? d.window : 0;
    v.R = log ? static_cast<int32_t>((d.flags >> 8) & 15u) : 0;
    v.plain = (d.flags & LS_PLAIN_UPDATE) ? 1 : 0;
    v.k16 = (d.flags & LS_LOG_BF16_K) ? 1 : 0;
    v.rec16 = (d.flags & LS_INT8_FP16_RECORDS) ? 1 : 0;
    v.cap = v.W + v.R;
    v.dl = d.gate == LS_GATE_PER_KEY ? kD : 1;
    v.lam_stride = d.gate == LS_GATE_PER_KEY ? v.cap * kD : (v.cap + 3) / 4 * 4;
    v.foldq = int8_mma_fold(&d) ? reinterpret_cast<int32_t*>(m + L.foldq) : nullptr;
    v.fold_grid = 1;
    v.mark = (d.flags & LS_CHECK_SLOTS) ? reinterpret_cast<int32_t*>(m + L.mark) : nullptr;
    return v;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int prepare_all() {
    // Idempotent per device; cheap enough to repeat at every pool creation.
    if (ls::prepare_eager_step_kernels() != cudaSuccess) return LS_ERR_CUDA;
    if (ls::prepare_log_step_kernels() != cudaSuccess) return LS_ERR_CUDA;
    if (ls::prepare_fold_kernels() != cudaSuccess) return LS_ERR_CUDA;
    if (ls::prepare_aux_kernels() != cudaSuccess) return LS_ERR_CUDA;
    if (ls::prepare_window_fold_kernels() != cudaSuccess) return LS_ERR_CUDA;
    if (ls::prepare_int8_step_kernels() != cudaSuccess) return LS_ERR_CUDA;
    return LS_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LS_OK : LS_ERR_CUDA; }

// Common checks of the calls that take a slot list.
int check_slot_list(const ls_pool* p, const int32_t* d_slots, int32_t n) {
    if (p == nullptr) return LS_ERR_INVALID;
    if (n < 0) return LS_ERR_INVALID;
    if (n == 0) return LS_OK;
    if (d_slots == nullptr) return LS_ERR_INVALID;
    if (!aligned(d_slots, 4)) return LS_ERR_ALIGN;
    if (n > p->desc.num_slots) return LS_ERR_SLOT;
    return LS_OK;
}

// LS_CHECK_SLOTS: the device check of a slot list for repeats, launched
// before the call that uses it.
int check_distinct(const ls_pool* p, const int32_t* d_slots, int32_t n, void* stream) {
    if (p->view.mark == nullptr) return LS_OK;
    return cuda_status(ls::launch_slot_check(p->view, d_slots, n, static_cast<cudaStream_t>(stream)));
}

ls::AuxArgs aux_args(const ls_pool* p, const int32_t* d_slots, int32_t n) {
    ls::AuxArgs a{};
    a.pv = p->view;
    a.slots = d_slots;
    a.n = n;
    return a;
}

// Validate one decode token's arguments and fill the kernel arguments
// (batch = 0 passes with nothing filled).
int step_args(ls_pool* pool, const int32_t* d_slot_idx, int32_t batch, const float* q,
              const float* k, const float* v, const float* log_decay, const float* beta,
              float* y, ls::StepArgs* a) {
    if (pool == nullptr || batch < 0) return LS_ERR_INVALID;
    if (batch == 0) return LS_OK;
    if (!d_slot_idx || !q || !k || !v || !log_decay || !beta || !y) return LS_ERR_INVALID;
    if (batch > pool->desc.num_slots) return LS_ERR_SLOT;
    if (static_cast<int64_t>(batch) * pool->desc.num_heads > 0x7fffffffLL) return LS_ERR_SIZE;
    const bool per_key = pool->desc.gate == LS_GATE_PER_KEY;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(y, 16) ||
        !aligned(log_decay, per_key ? 16 : 4) || !aligned(beta, 4) || !aligned(d_slot_idx, 4))
        return LS_ERR_ALIGN;
    a->pv = pool->view;
    a->slot_idx = d_slot_idx;
    a->batch = batch;
    a->q = q;
    a->k = k;
    a->v = v;
    a->lam = log_decay;
    a->beta = beta;
    a->y = y;
    return LS_OK;
}

// Split replay: coefficient entries per (request, head) row, the log
// capacity rounded up to whole streamed chunks.
int32_t split_stride(const ls_pool* p) {
    const int32_t cap = p->view.cap;
    return (cap + ls::kSplitEntries - 1) / ls::kSplitEntries * ls::kSplitEntries;
}

int launch_step(ls_pool* p, const ls::StepArgs& a, cudaStream_t s) {
    const ls_pool_desc& d = p->desc;
    const bool per_key = d.gate == LS_GATE_PER_KEY;
    if (d.variant == LS_EAGER_FP32) return cuda_status(ls::launch_eager_step(a, per_key, s));
    // deferred / INT8: one launch; a head whose window closes on this token
    // folds its log into the base inside the same kernel, or (INT8 with a
    // window-end queue) in the tensor-core fold launched right after it
    return cuda_status(ls::launch_log_step(a, d.variant == LS_WINDOW_INT8, per_key, s));
}

}  // namespace

int ls::pool_device(const ls_pool* p) { return p->device; }

extern "C" {

const char* ls_error_string(int status) {
    switch (status) {
        case LS_OK: return "ok";
        case LS_ERR_INVALID: return "invalid argument";
        case LS_ERR_ALIGN: return "misaligned pointer";
        case LS_ERR_SLOT: return "slot list longer than the pool";
        case LS_ERR_CUDA: return "CUDA runtime error";
        case LS_ERR_SIZE: return "unsupported size or buffer too small";
        default: return "unknown status";
    }
}

int ls_abi_version(void) { return LS_ABI_VERSION; }

int ls_pool_required_bytes(const ls_pool_desc* desc, size_t* bytes) {
    if (bytes == nullptr) return LS_ERR_INVALID;
    Layout L;
    const int rc = make_layout(desc, &L);
    if (rc != LS_OK) return rc;
    *bytes = L.total;
    return LS_OK;
}

int ls_pool_create(const ls_pool_desc* desc, void* dev_mem, size_t bytes, void* stream,
                   ls_pool** out) {
    if (out == nullptr || dev_mem == nullptr) return LS_ERR_INVALID;
    *out = nullptr;
    Layout L;
    const int rc = make_layout(desc, &L);
    if (rc != LS_OK) return rc;
    if (bytes < L.total) return LS_ERR_SIZE;
    if (!aligned(dev_mem, kAlign)) return LS_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LS_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return LS_ERR_CUDA;
    const int prc = prepare_all();
    if (prc != LS_OK) return prc;
    auto* p = new (std::nothrow) ls_pool;
    if (p == nullptr) return LS_ERR_INVALID;
    p->desc = *desc;
    p->mem = static_cast<unsigned char*>(dev_mem);
    p->bytes = bytes;
    p->view = make_view(*desc, L, p->mem);
    p->num_sms = sms > 0 ? sms : 1;
    p->device = dev;
    p->view.fold_grid = p->num_sms;
    if (cudaMemsetAsync(dev_mem, 0, L.total, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
        (p->view.R > 0 && ls::launch_init_comp(p->view, static_cast<cudaStream_t>(stream)) != cudaSuccess)) {
        delete p;
        return LS_ERR_CUDA;
    }
    *out = p;
    return LS_OK;
}

int ls_pool_destroy(ls_pool* pool) {
    delete pool;
    return LS_OK;
}

int ls_pool_load(ls_pool* pool, const int32_t* d_slots, int32_t n, const float* d_state,
                 void* stream) {
    int rc = check_slot_list(pool, d_slots, n);
    if (rc != LS_OK || n == 0) return rc;
    if (d_state == nullptr) return LS_ERR_INVALID;
    if (!aligned(d_state, 16)) return LS_ERR_ALIGN;
    if ((rc = check_distinct(pool, d_slots, n, stream)) != LS_OK) return rc;
    ls::AuxArgs a = aux_args(pool, d_slots, n);
    a.state_in = d_state;
    return cuda_status(ls::launch_load(a, pool->desc.variant == LS_WINDOW_INT8,
                                       is_log_variant(pool->desc.variant),
                                       static_cast<cudaStream_t>(stream)));
}

int ls_pool_reset_slots(ls_pool* pool, const int32_t* d_slots, int32_t n, void* stream) {
    int rc = check_slot_list(pool, d_slots, n);
    if (rc != LS_OK || n == 0) return rc;
    if ((rc = check_distinct(pool, d_slots, n, stream)) != LS_OK) return rc;
    return cuda_status(ls::launch_reset(aux_args(pool, d_slots, n),
                                        pool->desc.variant == LS_WINDOW_INT8,
                                        is_log_variant(pool->desc.variant),
                                        static_cast<cudaStream_t>(stream)));
}

int ls_decode_step(ls_pool* pool, const int32_t* d_slot_idx, int32_t batch, const float* q,
                   const float* k, const float* v, const float* log_decay, const float* beta,
                   float* y, void* stream) {
    ls::StepArgs a{};
    int rc = step_args(pool, d_slot_idx, batch, q, k, v, log_decay, beta, y, &a);
    if (rc != LS_OK || batch == 0) return rc;
    if ((rc = check_distinct(pool, d_slot_idx, batch, stream)) != LS_OK) return rc;
    return launch_step(pool, a, static_cast<cudaStream_t>(stream));
}

int ls_split_scratch_bytes(const ls_pool* pool, int32_t batch, size_t* bytes) {
    if (pool == nullptr || bytes == nullptr || batch < 0) return LS_ERR_INVALID;
    if (!is_log_variant(pool->desc.variant)) return LS_ERR_INVALID;
    *bytes = static_cast<size_t>(batch) * pool->desc.num_heads * split_stride(pool) * sizeof(float2);
    return LS_OK;
}

int ls_decode_step_split(ls_pool* pool, const int32_t* d_slot_idx, int32_t batch, const float* q,
                         const float* k, const float* v, const float* log_decay, const float* beta,
                         float* y, void* d_scratch, size_t scratch_bytes, void* stream) {
    ls::StepArgs a{};
    int rc = step_args(pool, d_slot_idx, batch, q, k, v, log_decay, beta, y, &a);
    if (rc != LS_OK || batch == 0) return rc;
    if (!is_log_variant(pool->desc.variant) || d_scratch == nullptr) return LS_ERR_INVALID;
    if (!aligned(d_scratch, 16)) return LS_ERR_ALIGN;
    size_t need = 0;
    ls_split_scratch_bytes(pool, batch, &need);
    if (scratch_bytes < need) return LS_ERR_SIZE;
    if ((rc = check_distinct(pool, d_slot_idx, batch, stream)) != LS_OK) return rc;
    a.coef = static_cast<float2*>(d_scratch);
    a.cstride = split_stride(pool);
    return cuda_status(ls::launch_log_step_split(a, pool->desc.variant == LS_WINDOW_INT8,
                                                 pool->desc.gate == LS_GATE_PER_KEY,
                                                 static_cast<cudaStream_t>(stream)));
}

int ls_step_staging_bytes(const ls_pool* pool, int32_t batch, size_t* bytes) {
    if (pool == nullptr || bytes == nullptr || batch < 0) return LS_ERR_INVALID;
    const size_t rows = static_cast<size_t>(batch) * pool->desc.num_heads;
    const size_t dl = pool->desc.gate == LS_GATE_PER_KEY ? kD : 1;
    size_t off = 0;
    off = align_up(off + static_cast<size_t>(batch) * 4);  // slots
    off = align_up(off + rows * kD * 4) * 1;               // q
    off = align_up(off + rows * kD * 4);                   // k
    off = align_up(off + rows * kD * 4);                   // v
    off = align_up(off + rows * dl * 4);                   // log_decay
    off = align_up(off + rows * 4);                        // beta
    off = align_up(off + rows * kD * 4);                   // y
    *bytes = off;
    return LS_OK;
}

int ls_decode_step_host(ls_pool* pool, const int32_t* h_slot_idx, int32_t batch, const float* h_q,
                        const float* h_k, const float* h_v, const float* h_log_decay,
                        const float* h_beta, float* h_y, void* d_staging, size_t staging_bytes,
                        void* stream) {
    if (pool == nullptr || batch < 0) return LS_ERR_INVALID;
    if (batch == 0) return LS_OK;
    if (!h_slot_idx || !h_q || !h_k || !h_v || !h_log_decay || !h_beta || !h_y || !d_staging)
        return LS_ERR_INVALID;
    if (!aligned(d_staging, kAlign)) return LS_ERR_ALIGN;
    size_t need = 0;
    int rc = ls_step_staging_bytes(pool, batch, &need);
    if (rc != LS_OK) return rc;
    if (staging_bytes < need) return LS_ERR_SIZE;
    const size_t rows = static_cast<size_t>(batch) * pool->desc.num_heads;
    const size_t dl = pool->desc.gate == LS_GATE_PER_KEY ? kD : 1;
    unsigned char* m = static_cast<unsigned char*>(d_staging);
    size_t off = 0;
    auto carve = [&](size_t n) {
        unsigned char* p = m + off;
        off = align_up(off + n);
        return p;
    };
    auto* d_slots = reinterpret_cast<int32_t*>(carve(static_cast<size_t>(batch) * 4));
    auto* d_q = reinterpret_cast<float*>(carve(rows * kD * 4));
    auto* d_k = reinterpret_cast<float*>(carve(rows * kD * 4));
    auto* d_v = reinterpret_cast<float*>(carve(rows * kD * 4));
    auto* d_l = reinterpret_cast<float*>(carve(rows * dl * 4));
    auto* d_b = reinterpret_cast<float*>(carve(rows * 4));
    auto* d_y = reinterpret_cast<float*>(carve(rows * kD * 4));
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
    if (cudaMemcpyAsync(d_slots, h_slot_idx, static_cast<size_t>(batch) * 4, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(d_q, h_q, rows * kD * 4, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(d_k, h_k, rows * kD * 4, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(d_v, h_v, rows * kD * 4, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(d_l, h_log_decay, rows * dl * 4, h2d, s) != cudaSuccess ||
        cudaMemcpyAsync(d_b, h_beta, rows * 4, h2d, s) != cudaSuccess)
        return LS_ERR_CUDA;
    rc = ls_decode_step(pool, d_slots, batch, d_q, d_k, d_v, d_l, d_b, d_y, stream);
    if (rc != LS_OK) return rc;
    if (cudaMemcpyAsync(h_y, d_y, rows * kD * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return LS_ERR_CUDA;
    return LS_OK;
}

int ls_window_commit(ls_pool* pool, const int32_t* d_slots, int32_t n, void* stream) {
    int rc = check_slot_list(pool, d_slots, n);
    if (rc != LS_OK || n == 0) return rc;
    const ls_pool_desc& d = pool->desc;
    if (!is_log_variant(d.variant)) return LS_OK;  // eager: always materialized
    if ((rc = check_distinct(pool, d_slots, n, stream)) != LS_OK) return rc;
    return cuda_status(ls::launch_fold(aux_args(pool, d_slots, n), d.variant == LS_WINDOW_INT8,
                                       d.gate == LS_GATE_PER_KEY, true,
                                       static_cast<cudaStream_t>(stream)));
}

int ls_pool_read(const ls_pool* pool, const int32_t* d_slots, int32_t n, float* d_state_out,
                 void* stream) {
    int rc = check_slot_list(pool, d_slots, n);
    if (rc != LS_OK || n == 0) return rc;
    if (d_state_out == nullptr) return LS_ERR_INVALID;
    if (!aligned(d_state_out, 16)) return LS_ERR_ALIGN;
    const ls_pool_desc& d = pool->desc;
    ls::AuxArgs a = aux_args(pool, d_slots, n);
    a.state_out = d_state_out;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!is_log_variant(d.variant)) return cuda_status(ls::launch_eager_read(a, s));
    return cuda_status(ls::launch_fold(a, d.variant == LS_WINDOW_INT8, d.gate == LS_GATE_PER_KEY,
                                       false, s));
}

int ls_pool_read_int8(const ls_pool* pool, const int32_t* d_slots, int32_t n, int8_t* d_codes,
                      float* d_scales, void* stream) {
    int rc = check_slot_list(pool, d_slots, n);
    if (rc != LS_OK || n == 0) return rc;
    if (pool->desc.variant != LS_WINDOW_INT8) return LS_ERR_INVALID;
    if (d_codes == nullptr || d_scales == nullptr) return LS_ERR_INVALID;
    if (!aligned(d_codes, 16) || !aligned(d_scales, 4)) return LS_ERR_ALIGN;
    ls::AuxArgs a = aux_args(pool, d_slots, n);
    a.codes_out = d_codes;
    a.scales_out = d_scales;
    return cuda_status(ls::launch_read_int8(a, static_cast<cudaStream_t>(stream)));
}

int ls_pool_read_int8_col_scales(const ls_pool* pool, const int32_t* d_slots, int32_t n,
                                 float* d_col_scales, void* stream) {
    int rc = check_slot_list(pool, d_slots, n);
    if (rc != LS_OK || n == 0) return rc;
    if (pool->view.colf == nullptr) return LS_ERR_INVALID;
    if (d_col_scales == nullptr) return LS_ERR_INVALID;
    if (!aligned(d_col_scales, 4)) return LS_ERR_ALIGN;
    ls::AuxArgs a = aux_args(pool, d_slots, n);
    a.scales_out = d_col_scales;
    return cuda_status(ls::launch_read_colf(a, static_cast<cudaStream_t>(stream)));
}

int ls_pool_read_compensators(const ls_pool* pool, const int32_t* d_slots, int32_t n,
                              float* d_k_out, float* d_u_out, void* stream) {
    int rc = check_slot_list(pool, d_slots, n);
    if (rc != LS_OK || n == 0) return rc;
    if (pool->view.R < 1) return LS_ERR_INVALID;
    if (d_k_out == nullptr || d_u_out == nullptr) return LS_ERR_INVALID;
    if (!aligned(d_k_out, 4) || !aligned(d_u_out, 4)) return LS_ERR_ALIGN;
    ls::AuxArgs a = aux_args(pool, d_slots, n);
    a.state_out = d_k_out;
    a.scales_out = d_u_out;
    return cuda_status(ls::launch_read_comp(a, static_cast<cudaStream_t>(stream)));
}

int ls_pool_read_log_meta(const ls_pool* pool, const int32_t* d_slots, int32_t n, int32_t* d_len,
                          float* d_lbar, void* stream) {
    int rc = check_slot_list(pool, d_slots, n);
    if (rc != LS_OK || n == 0) return rc;
    if (!is_log_variant(pool->desc.variant)) return LS_ERR_INVALID;
    if (d_len == nullptr) return LS_ERR_INVALID;
    if (!aligned(d_len, 4) || (d_lbar != nullptr && !aligned(d_lbar, 4))) return LS_ERR_ALIGN;
    ls::AuxArgs a = aux_args(pool, d_slots, n);
    a.len_out = d_len;
    a.lbar_out = d_lbar;
    return cuda_status(ls::launch_read_log_meta(a, static_cast<cudaStream_t>(stream)));
}

int ls_pool_status(ls_pool* pool, void* stream, int32_t* device_status) {
    if (pool == nullptr || device_status == nullptr) return LS_ERR_INVALID;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, pool->view.status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return LS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LS_ERR_CUDA;
    if (cudaMemsetAsync(pool->view.status, 0, sizeof(int32_t), s) != cudaSuccess) return LS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LS_ERR_CUDA;
    *device_status = v;
    return LS_OK;
}

}  // extern "C"
