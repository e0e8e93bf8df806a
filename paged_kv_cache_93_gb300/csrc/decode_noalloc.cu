// decode_noalloc.cu -- pkv_paged_decode_attn_noalloc: split-KV decode
// attention whose partial results live in a scratch array compiled into the
// library, so the call itself needs no device allocation at all.
//
// Who needs this: code that hands the library its inputs and outputs but may
// not create device buffers of its own -- for example a host framework that
// owns every byte of device memory through its own pool and forbids other
// components from calling cudaMalloc, a plugin loaded into such a framework,
// or a latency-critical loop where an allocation (and the synchronization it
// can imply) is not acceptable.  The regular entry point asks for a
// caller-provided workspace; these callers have nowhere to get one.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes.  Every
// GPU that loads the library holds it until the process exits.  All calls
// share it, so calls that overlap on the GPU (different streams, or graphs
// replayed concurrently) race on it; calls on one stream are ordered and safe.
// Nothing in it needs to start at zero: the split kernel writes every partial
// row (empty chunks included) before the merge reads it.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <mutex>

#include "pkv.h"

namespace {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_address[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in; the address must come from
// cudaGetSymbolAddress with the device current.  Looked up once per device.
void *scratch_address(int *status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = PKV_ERR_CUDA;
        return nullptr;
    }
    void *p = g_scratch_address[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    p = g_scratch_address[dev].load(std::memory_order_acquire);
    if (p) return p;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
        *status = PKV_ERR_CUDA;
        return nullptr;
    }
    g_scratch_address[dev].store(addr, std::memory_order_release);
    return addr;
}

}  // namespace

extern "C" int pkv_paged_decode_attn_noalloc(const pkv_cache_desc *cache, const float *q,
                                             int32_t batch, int32_t num_q_heads,
                                             const void *k_pool, const void *v_pool,
                                             const int32_t *block_tables, int32_t max_blocks,
                                             const int32_t *seq_lens, float scale,
                                             int32_t num_splits, float *out, float *lse,
                                             int32_t flags, pkv_stream_t stream) {
    if (!cache || batch < 0 || num_q_heads <= 0 || num_splits < 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    int32_t S = num_splits;
    if (S == 0) {
        const int64_t longest = int64_t(max_blocks > 0 ? max_blocks : 0) * cache->block_size;
        S = pkv_decode_auto_splits(cache, batch, num_q_heads,
                                   int32_t(longest < INT32_MAX ? longest : INT32_MAX));
    }
    // Partials [S][batch][heads][head_dim_v] + LSEs must fit the fixed scratch.
    if (pkv_decode_workspace_size(batch, num_q_heads, cache->head_dim_v, S) > kNoAllocScratchBytes)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    int status = PKV_OK;
    void *scratch = scratch_address(&status);
    if (!scratch) return status;
    return pkv_paged_decode_attn(cache, q, batch, num_q_heads, k_pool, v_pool, block_tables,
                                 max_blocks, seq_lens, scale, S, scratch, kNoAllocScratchBytes,
                                 out, lse, flags, stream);
}

extern "C" int pkv_paged_decode_attn_noalloc_e4m3(
    const pkv_cache_desc *cache, const float *q, int32_t batch, int32_t num_q_heads,
    const void *k_pool, const void *v_pool, const float *k_scale, const float *v_scale,
    const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens, float scale,
    int32_t num_splits, float *out, float *lse, int32_t flags, pkv_stream_t stream) {
    if (!cache || batch < 0 || num_q_heads <= 0 || num_splits < 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    int32_t S = num_splits;
    if (S == 0) {
        const int64_t longest = int64_t(max_blocks > 0 ? max_blocks : 0) * cache->block_size;
        S = pkv_decode_auto_splits_e4m3(cache, batch, num_q_heads,
                                        int32_t(longest < INT32_MAX ? longest : INT32_MAX));
    }
    if (pkv_decode_workspace_size(batch, num_q_heads, cache->head_dim_v, S) > kNoAllocScratchBytes)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    int status = PKV_OK;
    void *scratch = scratch_address(&status);
    if (!scratch) return status;
    return pkv_paged_decode_attn_e4m3(cache, q, batch, num_q_heads, k_pool, v_pool, k_scale,
                                      v_scale, block_tables, max_blocks, seq_lens, scale, S,
                                      scratch, kNoAllocScratchBytes, out, lse, flags, stream);
}
