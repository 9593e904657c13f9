// ls_static.cu -- ls_decode_step_split_static: the split-replay decode step
// with its coefficient scratch in a fixed device array, so that the call
// allocates nothing (no cudaMalloc, no allocating library call).
//
// The array is module-scope device storage: the CUDA runtime places one
// copy on every device the module is loaded on, zero-filled.  Its address
// is looked up once per device, with that device current, and kept.  A call
// is refused (LS_ERR_INVALID) unless the pool's device is the current one,
// so the array used is always the one on the device of the pool's memory.
#include <cuda_runtime.h>

#include <mutex>

#include "ls.h"
#include "ls_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_split_scratch[LS_SPLIT_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Address of g_split_scratch on the pool's device, which must be current.
int static_scratch(const ls_pool* pool, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LS_ERR_CUDA;
    if (dev != ls::pool_device(pool)) return LS_ERR_INVALID;
    if (dev < 0 || dev >= kMaxDevices) return LS_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_split_scratch) != cudaSuccess) return LS_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return LS_OK;
}

}  // namespace

extern "C" int ls_decode_step_split_static(ls_pool* pool, const int32_t* d_slot_idx, int32_t batch,
                                           const float* q, const float* k, const float* v,
                                           const float* log_decay, const float* beta, float* y,
                                           void* stream) {
    if (pool == nullptr || batch < 0) return LS_ERR_INVALID;
    if (batch == 0) return LS_OK;
    size_t need = 0;
    int rc = ls_split_scratch_bytes(pool, batch, &need);
    if (rc != LS_OK) return rc;
    if (need > LS_SPLIT_STATIC_SCRATCH_BYTES) return LS_ERR_SIZE;
    void* scratch = nullptr;
    if ((rc = static_scratch(pool, &scratch)) != LS_OK) return rc;
    // nothing in the array has to start at zero: every coefficient the step
    // reads was written by the prepare kernel of the same call (a log chunk
    // copies the coefficients of whole 6-entry groups, but the step reads
    // only those of the chunk's live entries)
    return ls_decode_step_split(pool, d_slot_idx, batch, q, k, v, log_decay, beta, y, scratch,
                                LS_SPLIT_STATIC_SCRATCH_BYTES, stream);
}
