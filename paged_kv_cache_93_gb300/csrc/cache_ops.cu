// cache_ops.cu -- the cache-maintenance half of libpkv: the device status
// word, slot mapping, kv_append, copy_blocks and the DCP interleaved slot
// mapping.  All of these move or index whole 16-byte vectors; none does
// floating-point arithmetic, so their results are bit-exact by construction.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

namespace {
// One status word per device (each device context holds its own copy).
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;
SymbolCache g_status_cache;
std::atomic<int> g_sm_count[kMaxDevices];
std::mutex g_setup_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(p);
        return static_cast<CtxGetCurrentFn>(nullptr);
    }();
    return fn;
}

// The calling thread's current CUDA context (the driver's handle), or
// nullptr when none is current or it cannot be read.
void *current_context() {
    CtxGetCurrentFn fn = ctx_get_current_fn();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}
}  // namespace

void *device_symbol_address(const void *symbol, SymbolCache &cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= SymbolCache::kMaxDevices)
        return nullptr;
    const void *ctx = current_context();
    const SymbolCache::Entry *e = cache.entry[dev].load(std::memory_order_acquire);
    if (e && ctx && e->ctx == ctx) return e->addr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    void *addr = nullptr;
    // The lookup makes the device's primary context current if no context was.
    if (cudaGetSymbolAddress(&addr, symbol) != cudaSuccess || !addr) return nullptr;
    ctx = current_context();
    e = cache.entry[dev].load(std::memory_order_acquire);
    if (!(e && e->ctx == ctx && e->addr == addr)) {
        // Entries are never freed: a reader may still hold the previous
        // one, and a process sees few contexts per device.
        cache.entry[dev].store(new SymbolCache::Entry{ctx, addr}, std::memory_order_release);
    }
    return addr;
}

uint32_t *status_word() {
    return static_cast<uint32_t *>(device_symbol_address(&g_status_word, g_status_cache));
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

bool valid_cache(const pkv_cache_desc *c) {
    return c && c->num_blocks > 0 && c->block_size >= 1 && c->block_size <= 256 &&
           c->num_kv_heads > 0 && c->head_dim_k > 0 && c->head_dim_v > 0 &&
           c->head_dim_k % 8 == 0 && c->head_dim_v % 8 == 0 && c->head_dim_k <= 1024 &&
           c->head_dim_v <= 1024;
}

int grid_for(int64_t work, int threads) {
    int64_t blocks = (work + threads - 1) / threads;
    int64_t cap = int64_t(sm_count()) * 8;
    return static_cast<int>(std::max<int64_t>(1, std::min(blocks, cap)));
}

// --------------------------------------------------------------- kernels

__global__ void slot_mapping_kernel(const int32_t *__restrict__ block_tables, int32_t batch,
                                    int32_t max_blocks, int32_t block_size, int32_t num_blocks,
                                    const int32_t *__restrict__ seq_ids,
                                    const int64_t *__restrict__ positions, int64_t num_tokens,
                                    int64_t *__restrict__ slots, uint32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < num_tokens;
         t += int64_t(gridDim.x) * blockDim.x) {
        const int32_t b = seq_ids[t];
        const int64_t pos = positions[t];
        int64_t slot = -1;
        if (b >= 0 && pos >= 0) {
            const int64_t lb = pos / block_size;
            if (b >= batch || lb >= max_blocks) {
                raise_status(status, PKV_DEV_TABLE_RANGE);
            } else {
                const int32_t phys = block_tables[int64_t(b) * max_blocks + lb];
                if (phys < 0 || phys >= num_blocks)
                    raise_status(status, PKV_DEV_BLOCK_ID);
                else
                    slot = int64_t(phys) * block_size + pos % block_size;
            }
        }
        slots[t] = slot;
    }
}

// One thread per 16-byte vector of a (token, KV head) row, K rows first then
// V rows.  Reads of k_new/v_new are contiguous across threads; each pool row
// is written by consecutive threads as one contiguous run.
__global__ void kv_append_kernel(uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                                 const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                 const int64_t *__restrict__ slots, int64_t num_tokens,
                                 int32_t num_kv_heads, int32_t block_size, int64_t num_slots,
                                 int32_t vk, int32_t vv, uint32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t per_token = int64_t(num_kv_heads) * (vk + vv);
    const int64_t total = num_tokens * per_token;
    for (int64_t u = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; u < total;
         u += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = u / per_token;
        int64_t r = u - t * per_token;
        const int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (r == 0) raise_status(status, PKV_DEV_SLOT);
            continue;
        }
        const int64_t block = slot / block_size, off = slot - block * block_size;
        if (r < int64_t(num_kv_heads) * vk) {
            const int64_t g = r / vk, c = r - g * vk;
            k_pool[((block * num_kv_heads + g) * block_size + off) * vk + c] =
                k_new[(t * num_kv_heads + g) * vk + c];
        } else {
            r -= int64_t(num_kv_heads) * vk;
            const int64_t g = r / vv, c = r - g * vv;
            v_pool[((block * num_kv_heads + g) * block_size + off) * vv + c] =
                v_new[(t * num_kv_heads + g) * vv + c];
        }
    }
}

// E4M3 pools: one thread per 8 elements of a (token, KV head) row (16 bytes of
// bf16 in, 8 bytes of codes out).  Element x of KV head g is stored as the
// code nearest to x / scale[g], the quotient rounded to binary32.
__global__ void kv_append_e4m3_kernel(uint2 *__restrict__ k_pool, uint2 *__restrict__ v_pool,
                                      const uint4 *__restrict__ k_new,
                                      const uint4 *__restrict__ v_new,
                                      const float *__restrict__ k_scale,
                                      const float *__restrict__ v_scale,
                                      const int64_t *__restrict__ slots, int64_t num_tokens,
                                      int32_t num_kv_heads, int32_t block_size, int64_t num_slots,
                                      int32_t vk, int32_t vv, uint32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t per_token = int64_t(num_kv_heads) * (vk + vv);
    const int64_t total = num_tokens * per_token;
    for (int64_t u = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; u < total;
         u += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = u / per_token;
        int64_t r = u - t * per_token;
        const int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (r == 0) raise_status(status, PKV_DEV_SLOT);
            continue;
        }
        const int64_t block = slot / block_size, off = slot - block * block_size;
        const bool is_k = r < int64_t(num_kv_heads) * vk;
        if (!is_k) r -= int64_t(num_kv_heads) * vk;
        const int32_t nv = is_k ? vk : vv;
        const int64_t g = r / nv, c = r - g * nv;
        const uint4 x = (is_k ? k_new : v_new)[(t * num_kv_heads + g) * nv + c];
        const float s = (is_k ? k_scale : v_scale)[g];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t codes[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t c01 = e4m3x2_from_f32(__fdiv_rn(bf16_lo_to_f32(w[2 * i]), s),
                                                 __fdiv_rn(bf16_hi_to_f32(w[2 * i]), s));
            const uint32_t c23 = e4m3x2_from_f32(__fdiv_rn(bf16_lo_to_f32(w[2 * i + 1]), s),
                                                 __fdiv_rn(bf16_hi_to_f32(w[2 * i + 1]), s));
            codes[i] = c01 | (c23 << 16);
        }
        (is_k ? k_pool : v_pool)[((block * num_kv_heads + g) * block_size + off) * nv + c] =
            make_uint2(codes[0], codes[1]);
    }
}

// grid.x = pair, grid.y splits a pair's K+V bytes.  Every CTA of a pair
// re-derives the same skip decision from the full pair list, so no CTA
// writes a destination that another pair reads or writes.
__global__ void copy_blocks_kernel(uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                                   const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                                   int32_t num_pairs, int32_t num_blocks, int64_t k_vecs,
                                   int64_t v_vecs, uint32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    const int32_t p = blockIdx.x;
    const int32_t s = src[p], d = dst[p];
    const bool in_range = s >= 0 && s < num_blocks && d >= 0 && d < num_blocks;
    int conflict = 0;
    for (int32_t q = threadIdx.x; q < num_pairs; q += blockDim.x)
        if (q != p && (dst[q] == d || src[q] == d)) conflict = 1;
    conflict = __syncthreads_or(conflict);
    if (!in_range || conflict) {
        if (blockIdx.y == 0 && threadIdx.x == 0)
            raise_status(status, in_range ? PKV_DEV_COPY_CONFLICT : PKV_DEV_BLOCK_ID);
        return;
    }
    const int64_t total = k_vecs + v_vecs;
    for (int64_t u = blockIdx.y * int64_t(blockDim.x) + threadIdx.x; u < total;
         u += int64_t(gridDim.y) * blockDim.x) {
        if (u < k_vecs)
            k_pool[int64_t(d) * k_vecs + u] = k_pool[int64_t(s) * k_vecs + u];
        else
            v_pool[int64_t(d) * v_vecs + (u - k_vecs)] = v_pool[int64_t(s) * v_vecs + (u - k_vecs)];
    }
}

// Token i: chunk c = i / I goes to partition r = c mod P as that
// partition's (c / P)-th chunk, so its local position is (c / P) * I + i mod I.
__global__ void interleave_slots_kernel(int64_t first_token, int64_t num_tokens, int32_t num_parts,
                                        int32_t interleave, int32_t block_size, int32_t num_blocks,
                                        const int32_t *__restrict__ part_tables, int32_t max_blocks,
                                        int64_t *__restrict__ slots, int32_t *__restrict__ parts,
                                        uint32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < num_tokens;
         t += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = first_token + t;
        const int64_t c = i / interleave;
        const int32_t r = static_cast<int32_t>(c % num_parts);
        const int64_t local = (c / num_parts) * interleave + (i - c * interleave);
        const int64_t lb = local / block_size;
        int64_t slot = -1;
        if (lb >= max_blocks) {
            raise_status(status, PKV_DEV_TABLE_RANGE);
        } else {
            const int32_t phys = part_tables[int64_t(r) * max_blocks + lb];
            if (phys < 0 || phys >= num_blocks)
                raise_status(status, PKV_DEV_BLOCK_ID);
            else
                slot = int64_t(phys) * block_size + (local - lb * block_size);
        }
        slots[t] = slot;
        if (parts) parts[t] = r;
    }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" const char *pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_SHAPE: return "unsupported or inconsistent shape";
        case PKV_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_DEVICE: return "device-side check failed";
        case PKV_ERR_NO_SPACE: return "no free blocks";
        case PKV_ERR_NOT_FOUND: return "unknown sequence";
        default: return "unknown status";
    }
}

extern "C" int pkv_device_status(uint32_t *flags, int reset, pkv_stream_t stream) {
    if (!flags) return PKV_ERR_INVALID_ARG;
    uint32_t *word = status_word();
    if (!word) return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (reset && cudaMemsetAsync(word, 0, sizeof(uint32_t), s) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    *flags = host;
    return PKV_OK;
}

extern "C" int pkv_slot_mapping(const pkv_cache_desc *cache, const int32_t *block_tables,
                                int32_t batch, int32_t max_blocks, const int32_t *seq_ids,
                                const int64_t *positions, int64_t num_tokens,
                                int64_t *slot_mapping, pkv_stream_t stream) {
    if (!valid_cache(cache) || batch < 0 || max_blocks < 0 || num_tokens < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!block_tables || !seq_ids || !positions || !slot_mapping) return PKV_ERR_INVALID_ARG;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int threads = 256;
    return launch_pdl(slot_mapping_kernel, dim3(grid_for(num_tokens, threads)), dim3(threads), 0,
                      reinterpret_cast<cudaStream_t>(stream), block_tables, batch, max_blocks,
                      cache->block_size, cache->num_blocks, seq_ids, positions, num_tokens,
                      slot_mapping, status);
}

extern "C" int pkv_kv_append(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                             const void *k_new, const void *v_new, const int64_t *slot_mapping,
                             int64_t num_tokens, pkv_stream_t stream) {
    if (!valid_cache(cache) || num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    // v_pool and v_new both NULL: the cache keeps no separate values (they
    // are the first head_dim_v dims of the key rows); only K is written.
    if (!k_pool || !k_new || !slot_mapping || !v_pool != !v_new) return PKV_ERR_INVALID_ARG;
    if (!v_pool && cache->head_dim_v > cache->head_dim_k) return PKV_ERR_SHAPE;
    if (!aligned16(k_pool) || !aligned16(k_new) || (v_pool && !aligned16(v_pool)) ||
        (v_new && !aligned16(v_new)))
        return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int32_t vk = cache->head_dim_k / 8;                      // 16-byte vectors
    const int32_t vv = v_pool ? cache->head_dim_v / 8 : 0;
    const int64_t work = num_tokens * cache->num_kv_heads * (vk + vv);
    const int threads = 256;
    return launch_pdl(kv_append_kernel, dim3(grid_for(work, threads)), dim3(threads), 0,
                      reinterpret_cast<cudaStream_t>(stream), static_cast<uint4 *>(k_pool),
                      static_cast<uint4 *>(v_pool), static_cast<const uint4 *>(k_new),
                      static_cast<const uint4 *>(v_new), slot_mapping, num_tokens,
                      cache->num_kv_heads, cache->block_size,
                      int64_t(cache->num_blocks) * cache->block_size, vk, vv, status);
}

extern "C" int pkv_kv_append_e4m3(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                                  const void *k_new, const void *v_new,
                                  const float *k_scale, const float *v_scale,
                                  const int64_t *slot_mapping, int64_t num_tokens,
                                  pkv_stream_t stream) {
    if (!valid_cache(cache) || num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_pool || !v_pool || !k_new || !v_new || !k_scale || !v_scale || !slot_mapping)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(k_pool) & 7) ||
        (reinterpret_cast<uintptr_t>(v_pool) & 7))
        return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int32_t vk = cache->head_dim_k / 8, vv = cache->head_dim_v / 8;   // 8-element groups
    const int64_t work = num_tokens * cache->num_kv_heads * (vk + vv);
    const int threads = 256;
    return launch_pdl(kv_append_e4m3_kernel, dim3(grid_for(work, threads)), dim3(threads), 0,
                      reinterpret_cast<cudaStream_t>(stream), static_cast<uint2 *>(k_pool),
                      static_cast<uint2 *>(v_pool), static_cast<const uint4 *>(k_new),
                      static_cast<const uint4 *>(v_new), k_scale, v_scale, slot_mapping,
                      num_tokens, cache->num_kv_heads, cache->block_size,
                      int64_t(cache->num_blocks) * cache->block_size, vk, vv, status);
}

namespace pkv {
namespace {
// Block copies of pools whose numbers take `elem_bytes` bytes each.
int copy_blocks_bytes(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                      const int32_t *src, const int32_t *dst, int32_t num_pairs,
                      pkv_stream_t stream, int elem_bytes);
}  // namespace
}  // namespace pkv

extern "C" int pkv_copy_blocks(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                               const int32_t *src, const int32_t *dst, int32_t num_pairs,
                               pkv_stream_t stream) {
    return pkv::copy_blocks_bytes(cache, k_pool, v_pool, src, dst, num_pairs, stream, 2);
}

extern "C" int pkv_copy_blocks_e4m3(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                                    const int32_t *src, const int32_t *dst, int32_t num_pairs,
                                    pkv_stream_t stream) {
    if (!v_pool) return PKV_ERR_INVALID_ARG;
    return pkv::copy_blocks_bytes(cache, k_pool, v_pool, src, dst, num_pairs, stream, 1);
}

namespace pkv {
namespace {
int copy_blocks_bytes(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                      const int32_t *src, const int32_t *dst, int32_t num_pairs,
                      pkv_stream_t stream, int elem_bytes) {
    if (!valid_cache(cache) || num_pairs < 0) return PKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PKV_OK;
    // v_pool NULL: the cache keeps no separate values; only K blocks are copied.
    if (!k_pool || !src || !dst) return PKV_ERR_INVALID_ARG;
    if (!v_pool && cache->head_dim_v > cache->head_dim_k) return PKV_ERR_SHAPE;
    if (!aligned16(k_pool) || (v_pool && !aligned16(v_pool))) return PKV_ERR_ALIGNMENT;
    if (num_pairs > 65535) return PKV_ERR_SHAPE;
    // 16-byte vectors per block
    const int64_t k_bytes =
        int64_t(cache->num_kv_heads) * cache->block_size * cache->head_dim_k * elem_bytes;
    const int64_t v_bytes =
        v_pool ? int64_t(cache->num_kv_heads) * cache->block_size * cache->head_dim_v * elem_bytes
               : 0;
    if (k_bytes % 16 || v_bytes % 16) return PKV_ERR_SHAPE;
    const int64_t k_vecs = k_bytes / 16, v_vecs = v_bytes / 16;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int threads = 256;
    // Enough CTAs per pair to cover the device a few times over.
    int64_t per_pair = (k_vecs + v_vecs + threads - 1) / threads;
    int64_t want = std::max<int64_t>(1, (int64_t(sm_count()) * 4 + num_pairs - 1) / num_pairs);
    dim3 grid(num_pairs, static_cast<unsigned>(std::min<int64_t>({per_pair, want, 65535})));
    return launch_pdl(copy_blocks_kernel, grid, dim3(threads), 0,
                      reinterpret_cast<cudaStream_t>(stream), static_cast<uint4 *>(k_pool),
                      static_cast<uint4 *>(v_pool), src, dst, num_pairs, cache->num_blocks, k_vecs,
                      v_vecs, status);
}
}  // namespace
}  // namespace pkv

extern "C" int64_t pkv_interleave_partition_len(int64_t num_tokens, int32_t num_parts,
                                                int32_t interleave, int32_t part) {
    if (num_tokens < 0 || num_parts <= 0 || interleave <= 0 || part < 0 || part >= num_parts)
        return -1;
    const int64_t cycle = int64_t(num_parts) * interleave;
    const int64_t full = num_tokens / cycle, rem = num_tokens - full * cycle;
    const int64_t tail = std::min<int64_t>(std::max<int64_t>(rem - int64_t(part) * interleave, 0),
                                           interleave);
    return full * interleave + tail;
}

extern "C" int pkv_interleave_slot_mapping(const pkv_cache_desc *cache, int64_t first_token,
                                           int64_t num_tokens, int32_t num_parts,
                                           int32_t interleave, const int32_t *part_block_tables,
                                           int32_t max_blocks, int64_t *slot_mapping,
                                           int32_t *part_of_token, pkv_stream_t stream) {
    if (!valid_cache(cache) || first_token < 0 || num_tokens < 0 || num_parts <= 0 ||
        interleave <= 0 || max_blocks < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!part_block_tables || !slot_mapping) return PKV_ERR_INVALID_ARG;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    const int threads = 256;
    return launch_pdl(interleave_slots_kernel, dim3(grid_for(num_tokens, threads)), dim3(threads),
                      0, reinterpret_cast<cudaStream_t>(stream), first_token, num_tokens,
                      num_parts, interleave, cache->block_size, cache->num_blocks,
                      part_block_tables, max_blocks, slot_mapping, part_of_token, status);
}
