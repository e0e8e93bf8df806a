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

#include <climits>
#include <cstdint>

#include "pkv.h"
#include "pkv_host.h"

namespace {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

pkv::SymbolCache g_scratch_cache;

// Device address of the scratch array in the current context.  In host code
// the array's name is only a host-side stand-in; the address comes from
// cudaGetSymbolAddress with the device current, looked up on the first call
// in each context and cached.
void *scratch_address(int *status) {
    void *p = pkv::device_symbol_address(&g_noalloc_scratch, g_scratch_cache);
    if (!p) *status = PKV_ERR_CUDA;
    return p;
}

int32_t table_span(const pkv_cache_desc *cache, int32_t max_blocks) {
    const int64_t longest = int64_t(max_blocks > 0 ? max_blocks : 0) * cache->block_size;
    return int32_t(longest < INT32_MAX ? longest : INT32_MAX);
}

}  // namespace

extern "C" int pkv_paged_decode_attn_noalloc(const pkv_cache_desc *cache, const float *q,
                                             int32_t batch, int32_t num_q_heads,
                                             const void *k_pool, const void *v_pool,
                                             const int32_t *block_tables, int32_t max_blocks,
                                             const int32_t *seq_lens, float scale,
                                             int32_t num_splits, float *out, float *lse,
                                             int32_t flags, pkv_stream_t stream) {
    // The regular entry point's checks first, so that a bad request gets the
    // status that call would give it.
    int st = pkv::validate_decode(cache, q, batch, num_q_heads, k_pool, v_pool, block_tables,
                                  max_blocks, seq_lens, num_splits, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (!out || !lse) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(out)) return PKV_ERR_ALIGNMENT;
    const int32_t S = num_splits != 0 ? num_splits
                                      : pkv_decode_auto_splits(cache, batch, num_q_heads,
                                                               table_span(cache, max_blocks));
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
    int st = pkv::validate_decode(cache, q, batch, num_q_heads, k_pool, v_pool, block_tables,
                                  max_blocks, seq_lens, num_splits, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (!v_pool || !k_scale || !v_scale || !out || !lse) return PKV_ERR_INVALID_ARG;
    if (!pkv::aligned16(out)) return PKV_ERR_ALIGNMENT;
    const int32_t S = num_splits != 0 ? num_splits
                                      : pkv_decode_auto_splits_e4m3(cache, batch, num_q_heads,
                                                                    table_span(cache, max_blocks));
    if (pkv_decode_workspace_size(batch, num_q_heads, cache->head_dim_v, S) > kNoAllocScratchBytes)
        return PKV_ERR_WORKSPACE_TOO_SMALL;
    int status = PKV_OK;
    void *scratch = scratch_address(&status);
    if (!scratch) return status;
    return pkv_paged_decode_attn_e4m3(cache, q, batch, num_q_heads, k_pool, v_pool, k_scale,
                                      v_scale, block_tables, max_blocks, seq_lens, scale, S,
                                      scratch, kNoAllocScratchBytes, out, lse, flags, stream);
}
