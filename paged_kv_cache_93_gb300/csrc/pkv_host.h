// pkv_host.h -- host-side declarations shared by the libpkv translation units
// (not part of the public C ABI).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// Per-device cache of a __device__ symbol's address, keyed on the CUDA
// context it was looked up in.
struct SymbolCache {
    static constexpr int kMaxDevices = 64;
    struct Entry {
        const void *ctx;
        void *addr;
    };
    std::atomic<const Entry *> entry[kMaxDevices] = {};
};

// Device address of the __device__ variable `symbol` in the calling
// thread's current context on the current device.  In host code such a
// variable's name is only a host-side stand-in; its device address comes
// from cudaGetSymbolAddress, looked up again whenever the current context
// is not the one cached (another context, or the device's primary context
// recreated after cudaDeviceReset).  nullptr if the CUDA runtime failed.
void *device_symbol_address(const void *symbol, SymbolCache &cache);

// Device address of the current device's status word.  nullptr if the CUDA
// runtime failed.
uint32_t *status_word();

// The argument and shape checks shared by every decode entry point (the
// statuses documented for pkv_paged_decode_attn); PKV_OK when they pass.
int validate_decode(const pkv_cache_desc *c, const float *q, int32_t batch, int32_t hq,
                    const void *k_pool, const void *v_pool, const int32_t *block_tables,
                    int32_t max_blocks, const int32_t *seq_lens, int32_t num_splits,
                    int32_t flags);

// Number of SMs of the current device (cached per device).
int sm_count();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// Launch with programmatic stream serialization, so the kernel may be
// scheduled while the previous kernel in the stream drains; every libpkv
// kernel calls pdl_wait() before it reads anything that kernel may write.
template <typename... Params, typename... Args>
int launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...));
}

// Launch the per-split decode kernels.  Arguments are already validated;
// `out_part`/`lse_part` are [S][B][Hq][Dv] / [S][B][Hq].
struct DecodeArgs {
    pkv_cache_desc cache;
    const float *q;
    int32_t batch, num_q_heads;
    const void *k_pool, *v_pool;
    const int32_t *block_tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    float scale;
    int32_t num_splits;
    float *out_part, *lse_part;
    uint32_t *status;
    cudaStream_t stream;
    // bf16 elements from one V row to the next: head_dim_v for a separate V
    // pool; head_dim_k when the values are the first head_dim_v dims of the
    // key rows (v_pool then points at the K pool).
    int32_t v_stride = 0;
    // Query tokens per sequence (T).  T > 1: q, out and lse hold batch * T
    // rows (sequence-major), and query token t of sequence b attends to the
    // first seq_lens[b] - T + 1 + t tokens.  Only the GQA TMA kernel reads
    // T; the other kernels are given one row per (sequence, token) instead.
    int32_t q_tokens = 1;
    // A sequence whose seq_len is below this sets PKV_DEV_SEQ_LEN (the
    // multi-token call: T, a sequence that cannot hold its T new tokens); 0
    // for the decode calls, where seq_len 0 is an empty row.
    int32_t flag_below = 0;
    // E4M3 pools: per-KV-head dequantisation scales (device, [num_kv_heads]).
    const float *k_scale = nullptr, *v_scale = nullptr;
    // Pipeline waits give up after this many nanoseconds (0: the kernels'
    // default limit).
    uint64_t wait_ns = 0;
    // Test control (PKV_DECODE_TEST_WITHHOLD): the producer issues no copies,
    // so the first wait for one runs out.  Read by the warp-level GQA kernel
    // and the tcgen05 large-group kernel only.
    int32_t withhold = 0;
};
bool tma_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads, int32_t q_tokens = 1);
// CTAs the warp-level GQA kernel keeps resident for the shape (one persistent grid).
int tma_resident_ctas(const pkv_cache_desc &c, int32_t num_q_heads, int32_t q_tokens = 1);
// 16 or 32 query rows per KV head (heads x query tokens; 32 as two head
// groups of 16), head dims 128: the tcgen05 form of the GQA kernel.
bool gqa_tc_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads, int32_t q_tokens);
int launch_decode_gqa_tc(const DecodeArgs &a);
// CTAs the tcgen05 GQA kernel keeps resident (one persistent grid).
int gqa_tc_resident_ctas();
// (sequence, KV head) items split into this many head groups of 16 rows
int gqa_tc_head_groups(const pkv_cache_desc &c, int32_t num_q_heads, int32_t q_tokens);
// E4M3 pools, 4, 8, 16 or 32 rows per KV head (query group x query tokens;
// 32 as two head groups of 16), head dims 128: the tcgen05 kernel with E4M3
// operands.
bool gqa_tc_e4m3_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads,
                                  int32_t q_tokens = 1);
// CTAs that kernel keeps resident for `group` rows per item (query group x
// query tokens).
int gqa_tc_e4m3_resident_ctas(int32_t group);
// Items per (sequence, KV head, split) for `group` rows: 2 at 32, else 1.
int gqa_tc_e4m3_head_groups(int32_t group);
int launch_decode_gqa_tc_e4m3(const DecodeArgs &a);
int launch_decode_tma(const DecodeArgs &a);
// Large query groups (G a multiple of 32, e.g. MLA-shaped 128 heads over one
// 576/512 latent head): tensor-core kernel with 32-head work items.
bool mla_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads);
int32_t mla_work_units(const pkv_cache_desc &c, int32_t batch, int32_t num_q_heads);
int launch_decode_mla(const DecodeArgs &a);
// Query groups that are a multiple of 64 heads on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators), 64-head work items.
bool mla_tc_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads);
int32_t mla_tc_work_units(const pkv_cache_desc &c, int32_t batch, int32_t num_q_heads);
int launch_decode_mla_tc(const DecodeArgs &a);
// Two problems over the same cache in one launch of that kernel (their work
// items walked together, the first problem's first); `second` supplies only
// its queries, tables, lengths, batch, heads, split count and partials.
int launch_decode_mla_tc_two(const DecodeArgs &first, const DecodeArgs &second);
// The same kernel over E4M3 pools (a.k_scale, a.v_scale set, values in
// their own pool): the codes are expanded to fp16 in shared memory, exactly.
bool mla_tc_e4m3_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads);
int launch_decode_mla_tc_e4m3(const DecodeArgs &a);
// The split kernel pkv_paged_decode_attn would launch for `a` (by shape and
// flags); writes a.out_part / a.lse_part as [S][batch][heads] partials.
int run_decode_split_kernel(const DecodeArgs &a, int32_t flags);
int launch_decode_generic(const DecodeArgs &a);
// The same over E4M3 pools (a.k_scale, a.v_scale set).
int launch_decode_generic_e4m3(const DecodeArgs &a);
int launch_lse_merge(int32_t num_parts, const float *out_part, const float *lse_part,
                     int64_t rows, int32_t head_dim_v, float *out, float *lse,
                     cudaStream_t stream);

}  // namespace pkv
