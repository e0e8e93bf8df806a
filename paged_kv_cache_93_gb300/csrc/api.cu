// api.cu -- C ABI entry points of the decode-attention path: argument
// validation, split selection, kernel choice and the split -> merge sequence.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

using namespace pkv;

namespace {
constexpr int32_t kMaxSplits = 256;
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
// PKV_DECODE_TEST_WITHHOLD is accepted only while a test has enabled it.
std::atomic<int> g_test_withhold_enabled{0};
// Pipeline wait limit under that control: long enough for any legitimate
// stall of a small test case, short enough to keep the test quick.
constexpr uint64_t kTestWaitNs = 1000000ull;
}  // namespace

namespace pkv {
int validate_decode(const pkv_cache_desc *c, const float *q, int32_t batch, int32_t hq,
                    const void *k_pool, const void *v_pool, const int32_t *block_tables,
                    int32_t max_blocks, const int32_t *seq_lens, int32_t num_splits,
                    int32_t flags) {
    const int32_t known = PKV_DECODE_GENERIC | PKV_DECODE_NO_TCGEN05 |
                          (g_test_withhold_enabled.load() ? PKV_DECODE_TEST_WITHHOLD : 0);
    if (!c || batch < 0 || hq <= 0 || max_blocks < 0 || num_splits < 0 ||
        num_splits > kMaxSplits || (flags & ~known) != 0)
        return PKV_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->block_size < 1 || c->block_size > 256 || c->num_kv_heads <= 0 ||
        c->head_dim_k <= 0 || c->head_dim_v <= 0)
        return PKV_ERR_INVALID_ARG;
    if (hq % c->num_kv_heads != 0 || c->head_dim_k % 8 != 0 || c->head_dim_v % 8 != 0 ||
        c->head_dim_k > 1024 || c->head_dim_v > 1024 || batch > 65535)
        return PKV_ERR_SHAPE;
    if (batch == 0) return PKV_OK;
    if (!q || !k_pool || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
    if (!v_pool && c->head_dim_v > c->head_dim_k) return PKV_ERR_SHAPE;   // values inside the keys
    if (!aligned16(q) || !aligned16(k_pool) || (v_pool && !aligned16(v_pool)))
        return PKV_ERR_ALIGNMENT;
    return PKV_OK;
}
}  // namespace pkv

namespace {

// The persistent GQA kernels' resident CTAs (tcgen05 and warp-level) take
// the (sequence, KV head [, head group], split) items in turn, an item costing its 128-token tiles
// plus about one tile of start-up.  Pick S for the least rounds x (tiles + 1)
// on sequences of the longest length; a tie goes to fewer splits (less to
// merge).
int32_t tc_splits(const pkv_cache_desc &c, int32_t batch, int32_t max_seq_len, int64_t ctas,
                  int32_t head_groups = 1) {
    const int64_t units = std::max<int64_t>(1, int64_t(batch) * c.num_kv_heads * head_groups);
    const int64_t L = std::max<int64_t>(1, max_seq_len);
    const int64_t s_max = std::min<int64_t>(kMaxSplits, (L + 127) / 128);
    int64_t best = 1, best_cost = INT64_MAX;
    for (int64_t s = 1; s <= s_max; ++s) {
        const int64_t chunk = 64 * ((L + 64 * s - 1) / (64 * s));
        const int64_t rounds = (units * s + ctas - 1) / ctas;
        const int64_t cost = rounds * ((chunk + 127) / 128 + 1);
        if (cost < best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return int32_t(best);
}

int32_t auto_splits(const pkv_cache_desc &c, int32_t batch, int32_t num_q_heads,
                    int32_t max_seq_len, int32_t q_tokens = 1) {
    if (gqa_tc_kernel_supports(c, num_q_heads, q_tokens))
        return tc_splits(c, batch, max_seq_len, gqa_tc_resident_ctas(),
                         gqa_tc_head_groups(c, num_q_heads, q_tokens));
    // The warp-level GQA kernel is a persistent grid too: an item count just
    // past its resident CTAs costs a second round (8 x 32K, 4 heads per KV
    // head: 10 splits 201 us, 8 splits 161 us).
    if (tma_kernel_supports(c, num_q_heads, q_tokens))
        return tc_splits(c, batch, max_seq_len, tma_resident_ctas(c, num_q_heads, q_tokens));
    // Enough (sequence, KV head [, head block], split) items for ~4 per SM
    // (8 for the tcgen05 kernel), each item at least 512 tokens long.
    int64_t units = int64_t(batch) * c.num_kv_heads;
    int64_t per_sm = 4;
    if (!tma_kernel_supports(c, num_q_heads)) {
        if (mla_tc_kernel_supports(c, num_q_heads)) {
            // one CTA per SM walks its items in turn: ~8 per SM evens out
            // the tail of unequal sequence lengths
            units = mla_tc_work_units(c, batch, num_q_heads);
            per_sm = 8;
        } else if (mla_kernel_supports(c, num_q_heads)) {
            units = mla_work_units(c, batch, num_q_heads);
        }
    }
    units = std::max<int64_t>(1, units);
    const int64_t want = (int64_t(sm_count()) * per_sm + units / 2) / units;
    const int64_t cap = std::max<int64_t>(1, (int64_t(max_seq_len) + 511) / 512);
    return int32_t(std::max<int64_t>(1, std::min<int64_t>({want, cap, kMaxSplits})));
}

// Where the values live: their own pool, or (v_pool NULL) the first
// head_dim_v dims of each key row.
void values_from(DecodeArgs &a) {
    if (a.v_pool) {
        a.v_stride = a.cache.head_dim_v;
    } else {
        a.v_pool = a.k_pool;
        a.v_stride = a.cache.head_dim_k;
    }
}

// The test control: the shape's split kernel with its copies withheld and a
// short wait limit.  Only the warp-level GQA kernel and the tcgen05
// large-group kernel read it; any other choice is refused before a launch.
int run_withheld(const DecodeArgs &in, int32_t flags) {
    DecodeArgs a = in;
    a.withhold = 1;
    a.wait_ns = kTestWaitNs;
    if (flags & PKV_DECODE_GENERIC) return PKV_ERR_INVALID_ARG;
    if (!(flags & PKV_DECODE_NO_TCGEN05) &&
        gqa_tc_kernel_supports(a.cache, a.num_q_heads, a.q_tokens))
        return PKV_ERR_INVALID_ARG;
    if (tma_kernel_supports(a.cache, a.num_q_heads, a.q_tokens)) return launch_decode_tma(a);
    if (!(flags & PKV_DECODE_NO_TCGEN05) && mla_tc_kernel_supports(a.cache, a.num_q_heads))
        return launch_decode_mla_tc(a);
    return PKV_ERR_INVALID_ARG;
}

int run_split_kernel(const DecodeArgs &a, int32_t flags) {
    if (flags & PKV_DECODE_TEST_WITHHOLD) return run_withheld(a, flags);
    if (!(flags & PKV_DECODE_GENERIC)) {
        if (!(flags & PKV_DECODE_NO_TCGEN05) &&
            gqa_tc_kernel_supports(a.cache, a.num_q_heads, a.q_tokens))
            return launch_decode_gqa_tc(a);
        if (tma_kernel_supports(a.cache, a.num_q_heads, a.q_tokens)) return launch_decode_tma(a);
        if (!(flags & PKV_DECODE_NO_TCGEN05) && mla_tc_kernel_supports(a.cache, a.num_q_heads))
            return launch_decode_mla_tc(a);
        if (mla_kernel_supports(a.cache, a.num_q_heads)) return launch_decode_mla(a);
    }
    return launch_decode_generic(a);
}

// The split kernel over E4M3 pools: the tcgen05 GQA kernel (4 to 32 rows
// per KV head, head dims 128), the tcgen05 large-group kernel (64 or more
// heads per KV head), else the CUDA-core kernel.  Under the test control
// only the large-group kernel runs (it reads it); anything else is refused.
int run_split_kernel_e4m3(const DecodeArgs &a, int32_t flags) {
    if (flags & PKV_DECODE_TEST_WITHHOLD) {
        if (flags != PKV_DECODE_TEST_WITHHOLD ||
            gqa_tc_e4m3_kernel_supports(a.cache, a.num_q_heads) ||
            !mla_tc_e4m3_kernel_supports(a.cache, a.num_q_heads))
            return PKV_ERR_INVALID_ARG;
        DecodeArgs w = a;
        w.withhold = 1;
        w.wait_ns = kTestWaitNs;
        return launch_decode_mla_tc_e4m3(w);
    }
    if (flags == 0 && gqa_tc_e4m3_kernel_supports(a.cache, a.num_q_heads))
        return launch_decode_gqa_tc_e4m3(a);
    if (flags == 0 && mla_tc_e4m3_kernel_supports(a.cache, a.num_q_heads))
        return launch_decode_mla_tc_e4m3(a);
    return launch_decode_generic_e4m3(a);
}

}  // namespace

namespace pkv {
int run_decode_split_kernel(const DecodeArgs &a, int32_t flags) { return run_split_kernel(a, flags); }
}  // namespace pkv

extern "C" int pkv_test_enable_withhold(int enable) {
    g_test_withhold_enabled.store(enable ? 1 : 0);
    return PKV_OK;
}

// Workspace layout: [partial outputs S x batch x heads x Dv fp32][partial
// LSEs S x batch x heads fp32], each region 256-byte aligned.
extern "C" size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                            int32_t head_dim_v, int32_t num_splits) {
    if (batch <= 0 || num_q_heads <= 0 || head_dim_v <= 0 || num_splits <= 1) return 0;
    const size_t rows = size_t(num_splits) * batch * num_q_heads;
    return align256(rows * head_dim_v * sizeof(float)) + align256(rows * sizeof(float));
}

extern "C" int32_t pkv_decode_auto_splits(const pkv_cache_desc *cache, int32_t batch,
                                          int32_t num_q_heads, int32_t max_seq_len) {
    if (!cache || cache->num_kv_heads <= 0 || num_q_heads <= 0) return 1;
    return auto_splits(*cache, batch, num_q_heads, max_seq_len);
}

extern "C" int pkv_paged_decode_attn_partial(const pkv_cache_desc *cache, const float *q,
                                             int32_t batch, int32_t num_q_heads,
                                             const void *k_pool, const void *v_pool,
                                             const int32_t *block_tables, int32_t max_blocks,
                                             const int32_t *seq_lens, float scale,
                                             int32_t num_splits, float *out_part,
                                             float *lse_part, int32_t flags,
                                             pkv_stream_t stream) {
    int st = validate_decode(cache, q, batch, num_q_heads, k_pool, v_pool, block_tables,
                             max_blocks, seq_lens, num_splits, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (num_splits < 1) return PKV_ERR_INVALID_ARG;
    if (!out_part || !lse_part) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out_part)) return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    DecodeArgs a{*cache, q, batch, num_q_heads, k_pool, v_pool, block_tables, max_blocks,
                 seq_lens, scale, num_splits, out_part, lse_part, status,
                 reinterpret_cast<cudaStream_t>(stream)};
    values_from(a);
    return run_split_kernel(a, flags);
}

extern "C" int32_t pkv_decode_auto_splits_e4m3(const pkv_cache_desc *cache, int32_t batch,
                                               int32_t num_q_heads, int32_t max_seq_len) {
    if (!cache || cache->num_kv_heads <= 0 || num_q_heads <= 0) return 1;
    if (!gqa_tc_e4m3_kernel_supports(*cache, num_q_heads))
        return auto_splits(*cache, batch, num_q_heads, max_seq_len);
    const int32_t group = num_q_heads / cache->num_kv_heads;
    return tc_splits(*cache, batch, max_seq_len, gqa_tc_e4m3_resident_ctas(group),
                     gqa_tc_e4m3_head_groups(group));
}

extern "C" int pkv_paged_decode_attn_e4m3(const pkv_cache_desc *cache, const float *q,
                                          int32_t batch, int32_t num_q_heads, const void *k_pool,
                                          const void *v_pool, const float *k_scale,
                                          const float *v_scale, const int32_t *block_tables,
                                          int32_t max_blocks, const int32_t *seq_lens,
                                          float scale, int32_t num_splits, void *workspace,
                                          size_t workspace_bytes, float *out, float *lse,
                                          int32_t flags, pkv_stream_t stream) {
    int st = validate_decode(cache, q, batch, num_q_heads, k_pool, v_pool, block_tables,
                             max_blocks, seq_lens, num_splits, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (!v_pool || !k_scale || !v_scale || !out || !lse) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out)) return PKV_ERR_ALIGNMENT;
    // the test control: only for shapes of the large-group kernel
    if ((flags & PKV_DECODE_TEST_WITHHOLD) &&
        (flags != PKV_DECODE_TEST_WITHHOLD || gqa_tc_e4m3_kernel_supports(*cache, num_q_heads) ||
         !mla_tc_e4m3_kernel_supports(*cache, num_q_heads)))
        return PKV_ERR_INVALID_ARG;
    // a tensor-core kernel where one takes the shape, the CUDA-core one
    // otherwise (or when a flag asks for it)
    auto launch = [&](const DecodeArgs &d) { return run_split_kernel_e4m3(d, flags); };
    int32_t S = num_splits;
    if (S == 0)
        S = pkv_decode_auto_splits_e4m3(
            cache, batch, num_q_heads,
            int32_t(std::min<int64_t>(int64_t(max_blocks) * cache->block_size, INT32_MAX)));
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, cache->head_dim_v, S);
    if (S > 1 && (!workspace || workspace_bytes < need)) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (S > 1 && !aligned16(workspace)) return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DecodeArgs a{*cache, q, batch, num_q_heads, k_pool, v_pool, block_tables, max_blocks,
                 seq_lens, scale, S, out, lse, status, s};
    a.v_stride = cache->head_dim_v;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    if (S == 1) return launch(a);
    const size_t rows = size_t(S) * batch * num_q_heads;
    char *ws = static_cast<char *>(workspace);
    a.out_part = reinterpret_cast<float *>(ws);
    a.lse_part = reinterpret_cast<float *>(ws + align256(rows * cache->head_dim_v * sizeof(float)));
    st = launch(a);
    if (st != PKV_OK) return st;
    return launch_lse_merge(S, a.out_part, a.lse_part, int64_t(batch) * num_q_heads,
                            cache->head_dim_v, out, lse, s);
}

extern "C" int pkv_paged_decode_attn_partial_e4m3(
    const pkv_cache_desc *cache, const float *q, int32_t batch, int32_t num_q_heads,
    const void *k_pool, const void *v_pool, const float *k_scale, const float *v_scale,
    const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens, float scale,
    int32_t num_splits, float *out_part, float *lse_part, int32_t flags, pkv_stream_t stream) {
    int st = validate_decode(cache, q, batch, num_q_heads, k_pool, v_pool, block_tables,
                             max_blocks, seq_lens, num_splits, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (num_splits < 1) return PKV_ERR_INVALID_ARG;
    if (flags & PKV_DECODE_TEST_WITHHOLD) return PKV_ERR_INVALID_ARG;
    if (!v_pool || !k_scale || !v_scale || !out_part || !lse_part) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out_part)) return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    DecodeArgs a{*cache, q, batch, num_q_heads, k_pool, v_pool, block_tables, max_blocks,
                 seq_lens, scale, num_splits, out_part, lse_part, status,
                 reinterpret_cast<cudaStream_t>(stream)};
    a.v_stride = cache->head_dim_v;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return run_split_kernel_e4m3(a, flags);
}

extern "C" int pkv_paged_decode_attn(const pkv_cache_desc *cache, const float *q, int32_t batch,
                                     int32_t num_q_heads, const void *k_pool, const void *v_pool,
                                     const int32_t *block_tables, int32_t max_blocks,
                                     const int32_t *seq_lens, float scale, int32_t num_splits,
                                     void *workspace, size_t workspace_bytes, float *out,
                                     float *lse, int32_t flags, pkv_stream_t stream) {
    int st = validate_decode(cache, q, batch, num_q_heads, k_pool, v_pool, block_tables,
                             max_blocks, seq_lens, num_splits, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (!out || !lse) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out)) return PKV_ERR_ALIGNMENT;
    int32_t S = num_splits;
    if (S == 0) {
        // Without a host copy of seq_lens, size the splits by the table width.
        S = auto_splits(*cache, batch, num_q_heads,
                        int32_t(std::min<int64_t>(int64_t(max_blocks) * cache->block_size,
                                                  INT32_MAX)));
    }
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, cache->head_dim_v, S);
    if (S > 1 && (!workspace || workspace_bytes < need)) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (S > 1 && !aligned16(workspace)) return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DecodeArgs a{*cache, q, batch, num_q_heads, k_pool, v_pool, block_tables, max_blocks,
                 seq_lens, scale, S, out, lse, status, s};
    values_from(a);
    if (S == 1) return run_split_kernel(a, flags);

    const size_t rows = size_t(S) * batch * num_q_heads;
    char *ws = static_cast<char *>(workspace);
    float *out_part = reinterpret_cast<float *>(ws);
    float *lse_part =
        reinterpret_cast<float *>(ws + align256(rows * cache->head_dim_v * sizeof(float)));
    a.out_part = out_part;
    a.lse_part = lse_part;
    // The split kernel lets the merge launch early (programmatic dependent
    // launch): the merge's CTAs wait on the device for the partials.
    st = run_split_kernel(a, flags);
    if (st != PKV_OK) return st;
    return launch_lse_merge(S, out_part, lse_part, int64_t(batch) * num_q_heads,
                            cache->head_dim_v, out, lse, s);
}

extern "C" int pkv_lse_merge(int32_t num_parts, const float *out_part, const float *lse_part,
                             int64_t rows, int32_t head_dim_v, float *out, float *lse,
                             pkv_stream_t stream) {
    if (num_parts <= 0 || rows < 0 || head_dim_v <= 0 || head_dim_v % 4 != 0 ||
        head_dim_v > 1024)
        return PKV_ERR_INVALID_ARG;
    if (rows == 0) return PKV_OK;
    if (!out_part || !lse_part || !out || !lse) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out_part) || !aligned16(out)) return PKV_ERR_ALIGNMENT;
    if (rows > int64_t(INT32_MAX)) return PKV_ERR_SHAPE;
    return launch_lse_merge(num_parts, out_part, lse_part, rows, head_dim_v, out, lse,
                            reinterpret_cast<cudaStream_t>(stream));
}

namespace {

constexpr int32_t kMaxQueryTokens = 64;

// Row r = b * T + t of a multi-token step reads sequence b's table and
// attends to its first seq_lens[b] - T + 1 + t tokens.  A sequence holding
// fewer than T tokens is flagged here (PKV_DEV_SEQ_LEN); its rows of
// negative length are treated as empty by the split kernel.
__global__ void multi_rows_kernel(const int32_t *__restrict__ block_tables,
                                  const int32_t *__restrict__ seq_lens, int32_t batch,
                                  int32_t tokens, int32_t max_blocks,
                                  int32_t *__restrict__ row_tables, int32_t *__restrict__ row_lens,
                                  uint32_t *__restrict__ status) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t rows = int64_t(batch) * tokens;
    const int64_t entries = rows * max_blocks;
    for (int64_t u = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; u < entries + rows;
         u += int64_t(gridDim.x) * blockDim.x) {
        if (u < entries) {
            const int64_t r = u / max_blocks, i = u - r * max_blocks;
            row_tables[u] = block_tables[(r / tokens) * max_blocks + i];
        } else {
            const int64_t r = u - entries, b = r / tokens;
            row_lens[r] = seq_lens[b] - (tokens - 1) + int32_t(r - b * tokens);
            if (r == b * tokens && seq_lens[b] < tokens) raise_status(status, PKV_DEV_SEQ_LEN);
        }
    }
}

struct MultiLayout {
    size_t tables, lens, partials, total;
};
MultiLayout multi_layout(int32_t batch, int32_t tokens, int32_t num_q_heads, int32_t head_dim_v,
                         int32_t max_blocks, int32_t num_splits) {
    MultiLayout m;
    const size_t rows = size_t(batch) * tokens;
    m.tables = 0;
    m.lens = align256(rows * size_t(max_blocks) * sizeof(int32_t));
    m.partials = m.lens + align256(rows * sizeof(int32_t));
    m.total = m.partials + pkv_decode_workspace_size(int32_t(rows), num_q_heads, head_dim_v,
                                                     num_splits);
    return m;
}

// Whether a GQA kernel takes a sequence's T query tokens as extra rows of one
// work item (the order run_split_kernel tries them in).
bool multi_folds(const pkv_cache_desc &c, int32_t num_q_heads, int32_t tokens, int32_t flags) {
    if (flags & PKV_DECODE_GENERIC) return false;
    return (!(flags & PKV_DECODE_NO_TCGEN05) && gqa_tc_kernel_supports(c, num_q_heads, tokens)) ||
           tma_kernel_supports(c, num_q_heads, tokens);
}

}  // namespace

extern "C" int32_t pkv_decode_multi_auto_splits(const pkv_cache_desc *cache, int32_t batch,
                                                int32_t tokens_per_seq, int32_t num_q_heads,
                                                int32_t max_seq_len, int32_t flags) {
    if (!cache || cache->num_kv_heads <= 0 || num_q_heads <= 0 || tokens_per_seq <= 0) return 1;
    // Work items are (sequence, KV head, split) when the GQA kernel takes the
    // T tokens as rows of one item; (sequence x token, KV head, split) otherwise.
    const bool folded = multi_folds(*cache, num_q_heads, tokens_per_seq, flags);
    return auto_splits(*cache, folded ? batch : batch * tokens_per_seq, num_q_heads,
                       max_seq_len, folded ? tokens_per_seq : 1);
}

extern "C" size_t pkv_decode_multi_workspace_size(int32_t batch, int32_t tokens_per_seq,
                                                  int32_t num_q_heads, int32_t head_dim_v,
                                                  int32_t max_blocks, int32_t num_splits) {
    if (batch <= 0 || tokens_per_seq <= 0 || num_q_heads <= 0 || head_dim_v <= 0 ||
        max_blocks < 0 || num_splits < 0 || int64_t(batch) * tokens_per_seq > 65535)
        return 0;
    return multi_layout(batch, tokens_per_seq, num_q_heads, head_dim_v, max_blocks,
                        std::max(num_splits, 1)).total;
}

extern "C" int pkv_paged_decode_attn_multi(const pkv_cache_desc *cache, const float *q,
                                           int32_t batch, int32_t tokens_per_seq,
                                           int32_t num_q_heads, const void *k_pool,
                                           const void *v_pool, const int32_t *block_tables,
                                           int32_t max_blocks, const int32_t *seq_lens,
                                           float scale, int32_t num_splits, void *workspace,
                                           size_t workspace_bytes, float *out, float *lse,
                                           int32_t flags, pkv_stream_t stream) {
    if (tokens_per_seq < 1 || tokens_per_seq > kMaxQueryTokens) return PKV_ERR_INVALID_ARG;
    if (flags & PKV_DECODE_TEST_WITHHOLD) return PKV_ERR_INVALID_ARG;
    if (batch > 0 && int64_t(batch) * tokens_per_seq > 65535) return PKV_ERR_SHAPE;
    const int32_t rows = batch * tokens_per_seq;
    int st = validate_decode(cache, q, rows, num_q_heads, k_pool, v_pool, block_tables,
                             max_blocks, seq_lens, num_splits, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (!out || !lse) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out)) return PKV_ERR_ALIGNMENT;
    int32_t S = num_splits;
    if (S == 0)
        S = pkv_decode_multi_auto_splits(
            cache, batch, tokens_per_seq, num_q_heads,
            int32_t(std::min<int64_t>(int64_t(max_blocks) * cache->block_size, INT32_MAX)), flags);
    const MultiLayout m = multi_layout(batch, tokens_per_seq, num_q_heads, cache->head_dim_v,
                                       max_blocks, S);
    if (!workspace || workspace_bytes < m.total) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const size_t prow = size_t(S) * rows * num_q_heads;
    float *out_part = reinterpret_cast<float *>(ws + m.partials);
    float *lse_part = reinterpret_cast<float *>(
        ws + m.partials + align256(prow * cache->head_dim_v * sizeof(float)));
    if (multi_folds(*cache, num_q_heads, tokens_per_seq, flags)) {
        // The GQA kernel takes the T query tokens as extra rows of each work
        // item (causal limits per row): every K/V tile is read once.
        DecodeArgs a{*cache, q, batch, num_q_heads, k_pool, v_pool, block_tables, max_blocks,
                     seq_lens, scale, S, out, lse, status, s};
        values_from(a);
        a.q_tokens = tokens_per_seq;
        a.flag_below = tokens_per_seq;
        if (S == 1) return run_split_kernel(a, flags);
        a.out_part = out_part;
        a.lse_part = lse_part;
        st = run_split_kernel(a, flags);
        if (st != PKV_OK) return st;
        return launch_lse_merge(S, out_part, lse_part, int64_t(rows) * num_q_heads,
                                cache->head_dim_v, out, lse, s);
    }
    // Otherwise one row per (sequence, token): T views of each table row.
    int32_t *row_tables = reinterpret_cast<int32_t *>(ws + m.tables);
    int32_t *row_lens = reinterpret_cast<int32_t *>(ws + m.lens);
    const int64_t work = int64_t(rows) * (int64_t(max_blocks) + 1);
    const int threads = 256;
    st = launch_pdl(multi_rows_kernel,
                    dim3(unsigned(std::min<int64_t>((work + threads - 1) / threads,
                                                    int64_t(sm_count()) * 8))),
                    dim3(threads), 0, s, block_tables, seq_lens, batch, tokens_per_seq,
                    max_blocks, row_tables, row_lens, status);
    if (st != PKV_OK) return st;
    DecodeArgs a{*cache, q, rows, num_q_heads, k_pool, v_pool, row_tables, max_blocks,
                 row_lens, scale, S, out, lse, status, s};
    values_from(a);
    if (S == 1) return run_split_kernel(a, flags);
    a.out_part = out_part;
    a.lse_part = lse_part;
    st = run_split_kernel(a, flags);
    if (st != PKV_OK) return st;
    return launch_lse_merge(S, out_part, lse_part, int64_t(rows) * num_q_heads,
                            cache->head_dim_v, out, lse, s);
}

extern "C" int32_t pkv_decode_multi_auto_splits_e4m3(const pkv_cache_desc *cache,
                                                     int32_t batch, int32_t tokens_per_seq,
                                                     int32_t num_q_heads, int32_t max_seq_len) {
    if (!cache || cache->num_kv_heads <= 0 || num_q_heads <= 0 || tokens_per_seq <= 0) return 1;
    if (gqa_tc_e4m3_kernel_supports(*cache, num_q_heads, tokens_per_seq))
        return tc_splits(*cache, batch, max_seq_len,
                         gqa_tc_e4m3_resident_ctas(num_q_heads / cache->num_kv_heads *
                                                   tokens_per_seq),
                         gqa_tc_e4m3_head_groups(num_q_heads / cache->num_kv_heads *
                                                 tokens_per_seq));
    return pkv_decode_auto_splits_e4m3(cache, batch * tokens_per_seq, num_q_heads, max_seq_len);
}

extern "C" int pkv_paged_decode_attn_multi_e4m3(
    const pkv_cache_desc *cache, const float *q, int32_t batch, int32_t tokens_per_seq,
    int32_t num_q_heads, const void *k_pool, const void *v_pool, const float *k_scale,
    const float *v_scale, const int32_t *block_tables, int32_t max_blocks,
    const int32_t *seq_lens, float scale, int32_t num_splits, void *workspace,
    size_t workspace_bytes, float *out, float *lse, int32_t flags, pkv_stream_t stream) {
    if (tokens_per_seq < 1 || tokens_per_seq > kMaxQueryTokens) return PKV_ERR_INVALID_ARG;
    if (flags & PKV_DECODE_TEST_WITHHOLD) return PKV_ERR_INVALID_ARG;
    if (batch > 0 && int64_t(batch) * tokens_per_seq > 65535) return PKV_ERR_SHAPE;
    const int32_t rows = batch * tokens_per_seq;
    int st = validate_decode(cache, q, rows, num_q_heads, k_pool, v_pool, block_tables,
                             max_blocks, seq_lens, num_splits, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (!v_pool || !k_scale || !v_scale || !out || !lse) return PKV_ERR_INVALID_ARG;
    if (!aligned16(out)) return PKV_ERR_ALIGNMENT;
    int32_t S = num_splits;
    if (S == 0)
        S = pkv_decode_multi_auto_splits_e4m3(
            cache, batch, tokens_per_seq, num_q_heads,
            int32_t(std::min<int64_t>(int64_t(max_blocks) * cache->block_size, INT32_MAX)));
    const MultiLayout m = multi_layout(batch, tokens_per_seq, num_q_heads, cache->head_dim_v,
                                       max_blocks, S);
    if (!workspace || workspace_bytes < m.total) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const size_t prow = size_t(S) * rows * num_q_heads;
    if (flags == 0 && gqa_tc_e4m3_kernel_supports(*cache, num_q_heads, tokens_per_seq)) {
        // The tensor-core kernel takes the T query tokens as rows of one work
        // item (causal limits per row): every tile is read once.
        DecodeArgs a{*cache, q, batch, num_q_heads, k_pool, v_pool, block_tables, max_blocks,
                     seq_lens, scale, S, out, lse, status, s};
        a.v_stride = cache->head_dim_v;
        a.k_scale = k_scale;
        a.v_scale = v_scale;
        a.q_tokens = tokens_per_seq;
        a.flag_below = tokens_per_seq;
        if (S == 1) return launch_decode_gqa_tc_e4m3(a);
        a.out_part = reinterpret_cast<float *>(ws + m.partials);
        a.lse_part = reinterpret_cast<float *>(ws + m.partials +
                                               align256(prow * cache->head_dim_v * sizeof(float)));
        st = launch_decode_gqa_tc_e4m3(a);
        if (st != PKV_OK) return st;
        return launch_lse_merge(S, a.out_part, a.lse_part, int64_t(rows) * num_q_heads,
                                cache->head_dim_v, out, lse, s);
    }
    // otherwise one row per (sequence, token): T views of each table row
    int32_t *row_tables = reinterpret_cast<int32_t *>(ws + m.tables);
    int32_t *row_lens = reinterpret_cast<int32_t *>(ws + m.lens);
    const int64_t work = int64_t(rows) * (int64_t(max_blocks) + 1);
    const int threads = 256;
    st = launch_pdl(multi_rows_kernel,
                    dim3(unsigned(std::min<int64_t>((work + threads - 1) / threads,
                                                    int64_t(sm_count()) * 8))),
                    dim3(threads), 0, s, block_tables, seq_lens, batch, tokens_per_seq,
                    max_blocks, row_tables, row_lens, status);
    if (st != PKV_OK) return st;
    DecodeArgs a{*cache, q, rows, num_q_heads, k_pool, v_pool, row_tables, max_blocks,
                 row_lens, scale, S, out, lse, status, s};
    a.v_stride = cache->head_dim_v;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    auto launch = [&](const DecodeArgs &d) { return run_split_kernel_e4m3(d, flags); };
    if (S == 1) return launch(a);
    a.out_part = reinterpret_cast<float *>(ws + m.partials);
    a.lse_part = reinterpret_cast<float *>(ws + m.partials +
                                           align256(prow * cache->head_dim_v * sizeof(float)));
    st = launch(a);
    if (st != PKV_OK) return st;
    return launch_lse_merge(S, a.out_part, a.lse_part, int64_t(rows) * num_q_heads,
                            cache->head_dim_v, out, lse, s);
}
