// cascade.cu -- decode attention of sequences that share a prefix, as a
// cascade: every query row of every sequence attends to the shared prefix
// blocks as the rows of ONE virtual sequence (so each staged prefix tile is
// multiplied by all the rows that need it, in items of 64 heads on the
// tcgen05 kernel), each sequence's rows attend to its own remaining tokens,
// and the two sets of partial results are merged by their LSEs.
//
//   prep   suffix tables (each table row past the prefix), suffix lengths,
//          the prefix length as a one-entry length array, a check that every
//          table begins with the shared prefix blocks, and (more than one KV
//          head) the query rows regrouped KV-head-major for the virtual
//          sequence
//   attend the prefix problem and the suffix problem in one persistent
//          launch of the tcgen05 kernel when it takes both shapes (the
//          suffix items fill the tail of the prefix items), else one
//          launch each
//   merge  per output row, the prefix partials and the suffix partials
#include <cuda_runtime.h>

#include <algorithm>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int32_t kMaxSplits = 256;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct CascadeLayout {
    size_t qv, stabs, slens, plen, pre_out, pre_lse, suf_out, suf_lse, total;
};

CascadeLayout cascade_layout(const pkv_cache_desc &c, int32_t batch, int32_t hq,
                             int32_t max_blocks, int32_t prefix_blocks, int32_t s1, int32_t s2) {
    CascadeLayout m;
    const size_t rows = size_t(batch) * hq;
    size_t at = 0;
    m.qv = at;
    at += c.num_kv_heads > 1 ? align256(rows * c.head_dim_k * sizeof(float)) : 0;
    m.stabs = at;
    at += align256(size_t(batch) * size_t(std::max(0, max_blocks - prefix_blocks)) *
                   sizeof(int32_t));
    m.slens = at;
    at += align256(size_t(batch) * sizeof(int32_t));
    m.plen = at;
    at += 256;
    m.pre_out = at;
    at += align256(size_t(s1) * rows * c.head_dim_v * sizeof(float));
    m.pre_lse = at;
    at += align256(size_t(s1) * rows * sizeof(float));
    m.suf_out = at;
    at += align256(size_t(s2) * rows * c.head_dim_v * sizeof(float));
    m.suf_lse = at;
    at += align256(size_t(s2) * rows * sizeof(float));
    m.total = at;
    return m;
}

// One grid-stride pass over four jobs: the suffix table rows, the suffix
// lengths (with the prefix length), the prefix check, and the regrouped
// query (row (g, b, j) of the virtual sequence = head g * G + j of sequence
// b).
__global__ void cascade_prep_kernel(const int32_t *__restrict__ prefix_table,
                                    int32_t prefix_blocks, const int32_t *__restrict__ tables,
                                    int32_t max_blocks, const int32_t *__restrict__ seq_lens,
                                    int32_t batch, int32_t block_size,
                                    const float *__restrict__ q, int32_t hq, int32_t hkv,
                                    int32_t dk, int32_t *__restrict__ stabs,
                                    int32_t *__restrict__ slens, int32_t *__restrict__ plen,
                                    float *__restrict__ qv, uint32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t sb = max_blocks > prefix_blocks ? max_blocks - prefix_blocks : 0;
    const int64_t n_tab = int64_t(batch) * sb;
    const int64_t n_chk = int64_t(batch) * prefix_blocks;
    const int64_t n_q = qv ? int64_t(batch) * hq * dk / 4 : 0;
    const int64_t P = int64_t(prefix_blocks) * block_size;
    const int G = hq / hkv;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t u = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; u < n_tab + n_chk + n_q + batch;
         u += stride) {
        if (u < n_tab) {
            const int64_t b = u / sb, i = u - b * sb;
            stabs[u] = tables[b * max_blocks + prefix_blocks + i];
        } else if (u < n_tab + n_chk) {
            const int64_t v = u - n_tab, b = v / prefix_blocks, i = v - b * prefix_blocks;
            if (tables[b * max_blocks + i] != prefix_table[i]) raise_status(status, PKV_DEV_PREFIX);
        } else if (u < n_tab + n_chk + n_q) {
            // virtual row r = (g * batch + b) * G + j  <-  q[b][g * G + j]
            const int64_t e = u - n_tab - n_chk, per_row = dk / 4;
            const int64_t r = e / per_row, c = e - r * per_row;
            const int64_t j = r % G, gb = r / G, b = gb % batch, g = gb / batch;
            reinterpret_cast<float4 *>(qv)[e] =
                reinterpret_cast<const float4 *>(q)[(b * hq + g * G + j) * per_row + c];
        } else {
            const int64_t b = u - n_tab - n_chk - n_q;
            const int64_t L = seq_lens[b];
            if (L < P) raise_status(status, PKV_DEV_SEQ_LEN);
            slens[b] = int32_t(L > P ? L - P : 0);
            if (b == 0) plen[0] = int32_t(P);
        }
    }
}

// Output row r = b * hq + h takes the prefix partials of virtual row
// (g * batch + b) * G + j (h = g * G + j) and its own suffix partials.
__global__ void cascade_merge_kernel(int32_t s1, const float *__restrict__ pre_out,
                                     const float *__restrict__ pre_lse, int32_t s2,
                                     const float *__restrict__ suf_out,
                                     const float *__restrict__ suf_lse, int32_t batch,
                                     int32_t hq, int32_t hkv, int32_t head_dim_v,
                                     float *__restrict__ out, float *__restrict__ lse) {
    pdl_wait();
    pdl_launch_dependents();
    const int tpr = head_dim_v / 4;
    const int64_t rows = int64_t(batch) * hq;
    const int64_t r = blockIdx.x * int64_t(blockDim.x / tpr) + threadIdx.x / tpr;
    const int c = threadIdx.x % tpr;
    if (r >= rows) return;
    const int64_t b = r / hq, h = r - b * hq;
    const int G = hq / hkv;
    const int64_t vr = (int64_t(h / G) * batch + b) * G + h % G;
    float M = -INFINITY, W = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool nan_part = false;
    for (int p0 = 0; p0 < s1 + s2; p0 += 8) {
        float l[8];
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int p = p0 + u;
            if (p < s1) {
                l[u] = pre_lse[int64_t(p) * rows + vr];
                x[u] = reinterpret_cast<const float4 *>(pre_out + (int64_t(p) * rows + vr) *
                                                                       head_dim_v)[c];
            } else if (p < s1 + s2) {
                const int64_t q = p - s1;
                l[u] = suf_lse[q * rows + r];
                x[u] = reinterpret_cast<const float4 *>(suf_out + (q * rows + r) * head_dim_v)[c];
            } else {
                l[u] = -INFINITY;
                x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float mc = M;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            nan_part |= l[u] != l[u];
            mc = fmaxf(mc, l[u]);
        }
        if (mc == -INFINITY) continue;
        const float rescale = expf(M - mc);
        W *= rescale;
        acc = make_float4(acc.x * rescale, acc.y * rescale, acc.z * rescale, acc.w * rescale);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float w = expf(l[u] - mc);
            if (w != 0.f) {
                W += w;
                acc.x = fmaf(w, x[u].x, acc.x); acc.y = fmaf(w, x[u].y, acc.y);
                acc.z = fmaf(w, x[u].z, acc.z); acc.w = fmaf(w, x[u].w, acc.w);
            }
        }
        M = mc;
    }
    float4 *orow = reinterpret_cast<float4 *>(out + r * head_dim_v);
    if (nan_part) {
        const float nan = __int_as_float(0x7fc00000);
        orow[c] = make_float4(nan, nan, nan, nan);
        if (c == 0) lse[r] = nan;
        return;
    }
    if (M == -INFINITY) {
        orow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c == 0) lse[r] = -INFINITY;
        return;
    }
    const float inv = 1.f / W;
    orow[c] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (c == 0) lse[r] = M + logf(W);
}

// Split counts when the caller passes 0.  The prefix: the usual rule for one
// sequence of batch x hq rows over the prefix tokens (on the tcgen05 kernel
// about 8 items per SM, all of one length).  The suffix: its items run after
// the prefix items in the same launch, so at most one per resident CTA
// (more would leave a tail of short items on some SMs), and chunks of at
// least 2,048 tokens (each item starts with a query load: 147 KB at Dk 576).
void resolve_splits(const pkv_cache_desc &c, int32_t batch, int32_t hq, int32_t max_blocks,
                    int32_t prefix_blocks, int32_t &s1, int32_t &s2) {
    const int64_t P = int64_t(prefix_blocks) * c.block_size;
    const int64_t Ls = int64_t(std::max(0, max_blocks - prefix_blocks)) * c.block_size;
    if (s1 == 0)
        s1 = P > 0 ? pkv_decode_auto_splits(&c, 1, batch * hq, int32_t(std::min<int64_t>(P, INT32_MAX)))
                   : 1;
    if (s2 == 0) {
        const int64_t units = std::max<int64_t>(
            1, mla_tc_kernel_supports(c, hq) ? mla_tc_work_units(c, batch, hq)
                                             : int64_t(batch) * c.num_kv_heads);
        const int64_t per_cta = std::max<int64_t>(1, sm_count() / units);
        s2 = int32_t(std::max<int64_t>(1, std::min<int64_t>({per_cta, (Ls + 2047) / 2048,
                                                             int64_t(kMaxSplits)})));
    }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_decode_cascade_splits(const pkv_cache_desc *cache, int32_t batch,
                                         int32_t num_q_heads, int32_t max_blocks,
                                         int32_t prefix_blocks, int32_t *prefix_splits,
                                         int32_t *suffix_splits) {
    if (!cache || !prefix_splits || !suffix_splits || batch < 0 || num_q_heads <= 0 ||
        cache->num_kv_heads <= 0 || cache->block_size <= 0 || prefix_blocks < 0 ||
        max_blocks < prefix_blocks || *prefix_splits < 0 || *suffix_splits < 0)
        return PKV_ERR_INVALID_ARG;
    resolve_splits(*cache, batch, num_q_heads, max_blocks, prefix_blocks, *prefix_splits,
                   *suffix_splits);
    return PKV_OK;
}

extern "C" size_t pkv_decode_cascade_workspace_size(const pkv_cache_desc *cache, int32_t batch,
                                                    int32_t num_q_heads, int32_t max_blocks,
                                                    int32_t prefix_blocks, int32_t prefix_splits,
                                                    int32_t suffix_splits) {
    if (!cache || batch <= 0 || num_q_heads <= 0 || cache->num_kv_heads <= 0 ||
        cache->head_dim_k <= 0 || cache->head_dim_v <= 0 || prefix_blocks < 0 ||
        max_blocks < prefix_blocks || prefix_splits < 0 || suffix_splits < 0)
        return 0;
    int32_t s1 = prefix_splits, s2 = suffix_splits;
    resolve_splits(*cache, batch, num_q_heads, max_blocks, prefix_blocks, s1, s2);
    return cascade_layout(*cache, batch, num_q_heads, max_blocks, prefix_blocks, s1, s2).total;
}

extern "C" int pkv_paged_decode_attn_cascade(
    const pkv_cache_desc *cache, const float *q, int32_t batch, int32_t num_q_heads,
    const void *k_pool, const void *v_pool, const int32_t *prefix_table, int32_t prefix_blocks,
    const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens, float scale,
    int32_t prefix_splits, int32_t suffix_splits, void *workspace, size_t workspace_bytes,
    float *out, float *lse, int32_t flags, pkv_stream_t stream) {
    if (flags & PKV_DECODE_TEST_WITHHOLD) return PKV_ERR_INVALID_ARG;
    int st = validate_decode(cache, q, batch, num_q_heads, k_pool, v_pool, block_tables,
                             max_blocks, seq_lens, 0, flags);
    if (st != PKV_OK || batch == 0) return st;
    if (prefix_blocks < 0 || prefix_blocks > max_blocks || prefix_splits < 0 ||
        suffix_splits < 0 || prefix_splits > kMaxSplits || suffix_splits > kMaxSplits ||
        (prefix_blocks > 0 && !prefix_table) || !out || !lse)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out)) return PKV_ERR_ALIGNMENT;
    if (int64_t(batch) * num_q_heads > 65535 * 64) return PKV_ERR_SHAPE;
    const pkv_cache_desc &c = *cache;
    int32_t s1 = prefix_splits, s2 = suffix_splits;
    resolve_splits(c, batch, num_q_heads, max_blocks, prefix_blocks, s1, s2);
    const CascadeLayout m = cascade_layout(c, batch, num_q_heads, max_blocks, prefix_blocks, s1, s2);
    if (!workspace || workspace_bytes < m.total) return PKV_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return PKV_ERR_ALIGNMENT;
    uint32_t *status = status_word();
    if (!status) return PKV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    int32_t *stabs = reinterpret_cast<int32_t *>(ws + m.stabs);
    int32_t *slens = reinterpret_cast<int32_t *>(ws + m.slens);
    int32_t *plen = reinterpret_cast<int32_t *>(ws + m.plen);
    float *qv = c.num_kv_heads > 1 ? reinterpret_cast<float *>(ws + m.qv) : nullptr;
    const int32_t hq = num_q_heads;

    // ---- prep
    {
        const int64_t work = int64_t(batch) * std::max(0, max_blocks - prefix_blocks) +
                             int64_t(batch) * prefix_blocks +
                             (qv ? int64_t(batch) * hq * c.head_dim_k / 4 : 0) + batch;
        const int threads = 256;
        const int grid = int(std::max<int64_t>(
            1, std::min<int64_t>((work + threads - 1) / threads, int64_t(sm_count()) * 8)));
        st = launch_pdl(cascade_prep_kernel, dim3(grid), dim3(threads), 0, s, prefix_table,
                        prefix_blocks, block_tables, max_blocks, seq_lens, batch, c.block_size, q,
                        hq, c.num_kv_heads, c.head_dim_k, stabs, slens, plen, qv, status);
        if (st != PKV_OK) return st;
    }

    // ---- the prefix problem: one virtual sequence of batch x hq rows over
    // the prefix blocks; the suffix problem: each sequence past the prefix
    DecodeArgs pre{c, qv ? qv : q, 1, batch * hq, k_pool, v_pool, prefix_table, prefix_blocks,
                   plen, scale, s1, reinterpret_cast<float *>(ws + m.pre_out),
                   reinterpret_cast<float *>(ws + m.pre_lse), status, s};
    DecodeArgs suf{c, q, batch, hq, k_pool, v_pool, stabs, max_blocks - prefix_blocks, slens,
                   scale, s2, reinterpret_cast<float *>(ws + m.suf_out),
                   reinterpret_cast<float *>(ws + m.suf_lse), status, s};
    if (v_pool) {
        pre.v_stride = suf.v_stride = c.head_dim_v;
    } else {
        pre.v_pool = suf.v_pool = k_pool;
        pre.v_stride = suf.v_stride = c.head_dim_k;
    }
    if (flags == 0 && mla_tc_kernel_supports(c, hq) && mla_tc_kernel_supports(c, batch * hq)) {
        st = launch_decode_mla_tc_two(pre, suf);
    } else {
        st = run_decode_split_kernel(pre, flags);
        if (st == PKV_OK) st = run_decode_split_kernel(suf, flags);
    }
    if (st != PKV_OK) return st;

    // ---- merge
    const int tpr = c.head_dim_v / 4;
    const int rows_per_cta = std::max(1, 256 / tpr);
    const int64_t rows = int64_t(batch) * hq;
    return launch_pdl(cascade_merge_kernel,
                      dim3(unsigned((rows + rows_per_cta - 1) / rows_per_cta)),
                      dim3(rows_per_cta * tpr), 0, s, s1,
                      reinterpret_cast<const float *>(ws + m.pre_out),
                      reinterpret_cast<const float *>(ws + m.pre_lse), s2,
                      reinterpret_cast<const float *>(ws + m.suf_out),
                      reinterpret_cast<const float *>(ws + m.suf_lse), batch, hq, c.num_kv_heads,
                      c.head_dim_v, out, lse);
}
