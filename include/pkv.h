/*
 * pkv.h -- C ABI of libpkv: paged KV-cache decode attention for GB300 (sm_103a).
 *
 * The operations follow these pages (cited by title and section):
 *   [PA]  "PagedAttentionとは？KVキャッシュを分割してLLMのメモリの無駄を減らす仕組み":
 *         "PagedAttentionはブロック表で論理順序と物理配置を分ける" (block tables),
 *         "要求の終了で空いたブロックを再利用する具体例" (allocation and reuse),
 *         "共通ブロックの共有とコピーオンライト" (ref counts, copy-on-write).
 *   [KVB] "1,000 人が同時に AI に質問したら、誰が最初に答えをもらうのか? KV キャッシュと
 *         continuous batching": "KV キャッシュは何を保持するのか?" (a decode step
 *         appends the new token's K/V, then attends over everything stored).
 *   [DCP] "なぜ長文LLMは遅くなるのか｜Decode Context ParallelismでKVキャッシュを分散する":
 *         interleaved assignment of tokens to partitions, the attention backend
 *         returning the softmax LSE, and the three-stage decode step whose last
 *         stage corrects the partial outputs with the shared LSEs and sums them.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    allocates no device memory.  Pointers must be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and returns a pkv_status.  A nonzero status from the host
 *    checks means nothing was launched.
 *  - Device addresses of the library's own device variables (the status
 *    word, the scratch of the _noalloc calls) are looked up per CUDA context
 *    and cached; a context destroyed and recreated under the same handle
 *    (cudaDeviceReset) is not noticed, so do not use the library across a
 *    device reset in one process.
 *  - Conditions only the device can see (a block id outside the pool, a slot
 *    out of range, a sequence longer than its table, overlapping copy pairs,
 *    a pipeline wait that gave up) never fault: the offending item is skipped
 *    and a bit is OR-ed into a per-device status word, read with
 *    pkv_device_status().
 *  - Cache layout (one layer): k_pool [num_blocks][num_kv_heads][block_size][head_dim_k]
 *    and v_pool [num_blocks][num_kv_heads][block_size][head_dim_v], bf16.  One
 *    (block, KV head) tile is contiguous.  Token j of sequence b lives in
 *    physical block block_tables[b][j / block_size] at offset j % block_size.
 *  - Values inside the keys (the latent layout of multi-head latent attention,
 *    where one cached row serves as the key and its first head_dim_v dims as
 *    the value): pass v_pool = NULL (and v_new = NULL to pkv_kv_append); the
 *    cache is then k_pool alone and head_dim_v <= head_dim_k.  The pages
 *    describe no such layout; it halves the bytes per token of the MLA shape.
 *  - Query head h uses KV head h / (num_q_heads / num_kv_heads).
 *  - Head dims: any multiple of 8 up to 1024 (which kernel runs a shape is
 *    listed with pkv_paged_decode_attn's flags); q, out and lse are fp32; lse
 *    is the natural log of sum_j exp(s_j) over the scaled scores
 *    s_j = scale * q . k_j.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pkv_stream_t; /* same type as cudaStream_t */

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,     /* null pointer, negative count, bad flag */
    PKV_ERR_SHAPE = -2,           /* unsupported or inconsistent dimensions */
    PKV_ERR_ALIGNMENT = -3,       /* a pointer is not 16-byte aligned */
    PKV_ERR_WORKSPACE_TOO_SMALL = -4,
    PKV_ERR_CUDA = -5,            /* a CUDA runtime call failed */
    PKV_ERR_DEVICE = -6,          /* the device status word holds an error bit */
    PKV_ERR_NO_SPACE = -7,        /* block manager: not enough free blocks */
    PKV_ERR_NOT_FOUND = -8        /* block manager: unknown sequence id */
} pkv_status;

/* Bits of the per-device status word (see pkv_device_status). */
#define PKV_DEV_BLOCK_ID      0x1u  /* a block id outside [0, num_blocks) was met */
#define PKV_DEV_SLOT          0x2u  /* a slot outside [0, num_blocks*block_size) */
#define PKV_DEV_SEQ_LEN       0x4u  /* seq_len < 0 or > max_blocks * block_size */
#define PKV_DEV_COPY_CONFLICT 0x8u  /* copy pairs share a destination, or a
                                       destination is another pair's source */
#define PKV_DEV_TIMEOUT       0x10u /* a pipeline wait gave up (library bug) */
#define PKV_DEV_TABLE_RANGE   0x20u /* a position past the end of its table row */
#define PKV_DEV_PREFIX        0x40u /* cascade: a table that does not begin with the
                                       shared prefix blocks */

/* Shape of one layer's paged KV cache. */
typedef struct pkv_cache_desc {
    int32_t num_blocks;
    int32_t block_size;   /* tokens per block, 1..256 */
    int32_t num_kv_heads;
    int32_t head_dim_k;
    int32_t head_dim_v;
} pkv_cache_desc;

/* Human-readable name of a pkv_status value. */
const char *pkv_status_string(int status);

/* Reads the current device's status word into *flags after synchronizing
 * `stream`; clears it when `reset` is nonzero.  Returns PKV_OK, or
 * PKV_ERR_CUDA if the copy failed.  The word is shared by every call on the
 * device; it is never cleared implicitly. */
int pkv_device_status(uint32_t *flags, int reset, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_slot_mapping -- [PA] "PagedAttentionはブロック表で論理順序と物理配置を分ける":
 * the slot (physical block * block_size + offset) of logical position
 * positions[t] of sequence seq_ids[t]:
 *     slot = block_tables[seq][pos / block_size] * block_size + pos % block_size.
 * seq_ids [T] int32, positions [T] int64, block_tables [batch][max_blocks] int32,
 * slot_mapping [T] int64 (output).  A negative seq id or position gives -1
 * (padding).  A position past the table row or a block id outside the pool
 * gives -1 and sets PKV_DEV_TABLE_RANGE / PKV_DEV_BLOCK_ID.
 * ------------------------------------------------------------------------- */
int pkv_slot_mapping(const pkv_cache_desc *cache, const int32_t *block_tables,
                     int32_t batch, int32_t max_blocks, const int32_t *seq_ids,
                     const int64_t *positions, int64_t num_tokens, int64_t *slot_mapping,
                     pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_kv_append -- [KVB] "KV キャッシュは何を保持するのか?": write each new token's
 * key and value into the cache.  Token t's K row for KV head g
 * (k_new[t][g][0..head_dim_k)) goes to k_pool[slot / bs][g][slot % bs][:], and
 * likewise for V, with slot = slot_mapping[t].  k_new [T][num_kv_heads][head_dim_k]
 * and v_new [T][num_kv_heads][head_dim_v] bf16; slot_mapping [T] int64.
 * Negative slots are skipped (padding); slots >= num_blocks * block_size are
 * skipped and set PKV_DEV_SLOT.  Two tokens with the same slot race.  With
 * v_pool and v_new both NULL (values inside the keys) only K is written; one
 * of the two NULL is PKV_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
int pkv_kv_append(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                  const void *k_new, const void *v_new, const int64_t *slot_mapping,
                  int64_t num_tokens, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_copy_blocks -- [PA] "共通ブロックの共有とコピーオンライト": before a sequence
 * writes into a block it shares, the block is duplicated (and the caller then
 * points that sequence's table at the copy).  For each i < num_pairs, every KV
 * head's K and V tile of block src[i] is copied to block dst[i].  src, dst:
 * [num_pairs] int32 device arrays.  A pair whose ids are out of range sets
 * PKV_DEV_BLOCK_ID; a pair whose destination is also another pair's
 * destination or any pair's source sets PKV_DEV_COPY_CONFLICT; such pairs are
 * skipped, so the others never race with them.  v_pool NULL (values inside
 * the keys): only the K tiles are copied.
 * ------------------------------------------------------------------------- */
int pkv_copy_blocks(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                    const int32_t *src, const int32_t *dst, int32_t num_pairs,
                    pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 cache -- [DCP] counts a cached number's bytes by data type (FP8: one
 * byte) and names storing the KV cache in a low-precision type such as FP8
 * as the way to shrink each token's bytes; [PA] "Continuous Batching・prefix
 * caching・量子化との違い": quantisation changes the stored representation, so
 * its effect on accuracy has to be checked.  The pages fix no format; here
 * FP8 is E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, S.1111.111 = NaN, largest finite 448).  E4M3 pools have the
 * bf16 pools' shapes with one-byte elements (uint8 codes, 8-byte aligned).
 * Each KV head g has dequantisation scales k_scale[g] and v_scale[g] (fp32
 * device arrays [num_kv_heads], caller-owned, positive and finite): code c
 * of KV head g reads back as value(c) * scale[g].  Scales are chosen by the
 * caller (e.g. a head's largest magnitude / 448) and stay fixed while a
 * pool holds values quantised with them.
 *
 * pkv_kv_append_e4m3: pkv_kv_append into E4M3 pools.  k_new, v_new bf16 as
 * for pkv_kv_append (16-byte aligned); element x of KV head g is stored as
 * the code nearest to x / scale[g] -- the quotient rounded to binary32, a
 * tie going to the even code, magnitudes of 448 and beyond stored as +-448.
 * head_dim_k and head_dim_v multiples of 8.  Slots as pkv_kv_append.
 *
 * pkv_copy_blocks_e4m3: pkv_copy_blocks for E4M3 pools (both pools given;
 * num_kv_heads * block_size * head_dim a multiple of 16, else PKV_ERR_SHAPE).
 * ------------------------------------------------------------------------- */
int pkv_kv_append_e4m3(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                       const void *k_new, const void *v_new, const float *k_scale,
                       const float *v_scale, const int64_t *slot_mapping, int64_t num_tokens,
                       pkv_stream_t stream);

int pkv_copy_blocks_e4m3(const pkv_cache_desc *cache, void *k_pool, void *v_pool,
                         const int32_t *src, const int32_t *dst, int32_t num_pairs,
                         pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_interleave_slot_mapping -- [DCP] interleaved assignment: the KV of token i
 * belongs to partition (i / interleave) mod num_parts, and each partition
 * keeps its tokens in their original order.  For tokens
 * i = first_token .. first_token + num_tokens - 1 this writes the slot of
 * token i inside its partition's table: part_block_tables [num_parts][max_blocks]
 * int32 (each partition's table over a shared pool), slot_mapping [num_tokens]
 * int64, and, when part_of_token is not NULL, the partition [num_tokens] int32.
 * A local position past the partition's table gives -1 and sets
 * PKV_DEV_TABLE_RANGE.
 * ------------------------------------------------------------------------- */
int pkv_interleave_slot_mapping(const pkv_cache_desc *cache, int64_t first_token,
                                int64_t num_tokens, int32_t num_parts, int32_t interleave,
                                const int32_t *part_block_tables, int32_t max_blocks,
                                int64_t *slot_mapping, int32_t *part_of_token,
                                pkv_stream_t stream);

/* Host helper: how many of tokens 0..num_tokens-1 partition `part` holds
 * under the same rule.  Returns -1 on invalid arguments. */
int64_t pkv_interleave_partition_len(int64_t num_tokens, int32_t num_parts,
                                     int32_t interleave, int32_t part);

/* ---------------------------------------------------------------------------
 * Decode attention.  [KVB] the new token's query is compared with the keys
 * of all stored tokens and weights their values; [PA] the KV is read through
 * the block table and the result is the same as for contiguous storage;
 * [DCP] the backend also returns the softmax LSE.  For sequence b, query head
 * h, KV head g = h / (num_q_heads / num_kv_heads) and j < seq_lens[b]:
 *     s_j = scale * sum_d q[b][h][d] * K_j[d]
 *     out[b][h][:] = sum_j e^{s_j} V_j / sum_j e^{s_j},  lse[b][h] = ln sum_j e^{s_j}
 * q [batch][num_q_heads][head_dim_k] fp32; out [batch][num_q_heads][head_dim_v]
 * fp32; lse [batch][num_q_heads] fp32.  seq_lens[b] == 0 gives out = 0 and
 * lse = -inf.  A seq_len outside [0, max_blocks * block_size] is treated as 0
 * and sets PKV_DEV_SEQ_LEN.  A table entry outside [0, num_blocks) is never
 * dereferenced: its tokens read some in-pool block instead, the row's result
 * is unspecified, and PKV_DEV_BLOCK_ID is set.  v_pool NULL: V_j is the first
 * head_dim_v dims of K_j (head_dim_v > head_dim_k is PKV_ERR_SHAPE).
 *
 * Split-KV: with num_splits = S > 1 each sequence's tokens are cut into S
 * contiguous chunks, chunk s covering [s*C_b, min(seq_lens[b], (s+1)*C_b)) with
 * C_b = 64 * ceil(seq_lens[b] / (64 * S)); each chunk's partial (out, lse) is
 * computed separately and the partials are merged exactly as pkv_lse_merge
 * does.  num_splits = 0 picks S from the batch, the heads and the SM count.
 * S must be <= 256.  A chunk whose kernel gave up on a pipeline wait
 * (PKV_DEV_TIMEOUT) is abandoned: its rows come back NaN, output and LSE, and
 * the merge passes a NaN partial on as a NaN row.  The partials live in `workspace`, which must hold at
 * least pkv_decode_workspace_size(batch, num_q_heads, head_dim_v, S) bytes
 * (0 when S == 1; `workspace` may then be NULL).  Its contents on entry do
 * not matter.
 *
 * flags: 0 = choose the kernel by shape: the TMA + tensor-core GQA kernel
 * for head_dim_k == head_dim_v in {64, 128}, query groups of 1, 2, 4, 8 or
 * 16 and power-of-two block sizes >= 8; for query groups that are a multiple
 * of 64 (MLA-shaped, e.g. 128 heads over one 576/512 latent head) with
 * head_dim_k a multiple of 64 up to 576, head_dim_v a multiple of 128 up to
 * 512 and power-of-two block sizes 64..256, the tcgen05 kernel (5th-
 * generation tensor cores, accumulators in tensor memory); for other query
 * groups that are a multiple of 32 (head dims multiples of 64, head_dim_v
 * <= 512, power-of-two block sizes >= 32) the warp-level-MMA large-group
 * kernel; the generic CUDA-core kernel otherwise.  PKV_DECODE_GENERIC forces
 * the generic kernel.  Query groups of 16 or 32 (or 16 or 32 rows of heads x
 * query tokens in pkv_paged_decode_attn_multi; 32 as two work items of 16
 * heads' rows that read the same tiles) with head dims 128 and power-of-two
 * block sizes >= 16 run on a tcgen05 form of the GQA kernel.
 * PKV_DECODE_NO_TCGEN05 passes over both tcgen05 kernels (the warp-level-MMA
 * kernels take their shapes).
 * ------------------------------------------------------------------------- */
#define PKV_DECODE_GENERIC 0x1
#define PKV_DECODE_NO_TCGEN05 0x2

/* ---------------------------------------------------------------------------
 * Test control of the failure path (the pages have no counterpart; it exists
 * so that the bounded pipeline waits can be made to run out on purpose,
 * without any fault).  After pkv_test_enable_withhold(1), flag
 * PKV_DECODE_TEST_WITHHOLD makes pkv_paged_decode_attn (and its _partial
 * and _noalloc forms, and pkv_paged_decode_attn_e4m3 and its _noalloc form
 * for query groups of 64+ heads) run the shape's split kernel with its copy producer
 * issuing no copy at all and every pipeline wait limited to 1 ms: the first
 * wait for a copy runs out, the kernel sets PKV_DEV_TIMEOUT, every role of
 * each CTA leaves its loop with nothing in flight, and every row of the call
 * comes back NaN (output and LSE), as any abandoned chunk does.  Only the
 * warp-level GQA kernel and the tcgen05 large-group kernel (both of its
 * modes) take the flag;
 * for other shapes, the other entry points, or while it is not enabled
 * (pkv_test_enable_withhold(0), the default) it is PKV_ERR_INVALID_ARG.
 * Returns PKV_OK.
 * ------------------------------------------------------------------------- */
#define PKV_DECODE_TEST_WITHHOLD 0x100
int pkv_test_enable_withhold(int enable);

size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t head_dim_v,
                                 int32_t num_splits);

/* The split count num_splits = 0 resolves to for this batch on the current device. */
int32_t pkv_decode_auto_splits(const pkv_cache_desc *cache, int32_t batch,
                               int32_t num_q_heads, int32_t max_seq_len);

int pkv_paged_decode_attn(const pkv_cache_desc *cache, const float *q, int32_t batch,
                          int32_t num_q_heads, const void *k_pool, const void *v_pool,
                          const int32_t *block_tables, int32_t max_blocks,
                          const int32_t *seq_lens, float scale, int32_t num_splits,
                          void *workspace, size_t workspace_bytes, float *out, float *lse,
                          int32_t flags, pkv_stream_t stream);

/* The per-chunk partials themselves: out_part [S][batch][num_q_heads][head_dim_v]
 * and lse_part [S][batch][num_q_heads], chunks as above; an empty chunk gives
 * out = 0, lse = -inf.  pkv_lse_merge of these equals pkv_paged_decode_attn. */
int pkv_paged_decode_attn_partial(const pkv_cache_desc *cache, const float *q, int32_t batch,
                                  int32_t num_q_heads, const void *k_pool, const void *v_pool,
                                  const int32_t *block_tables, int32_t max_blocks,
                                  const int32_t *seq_lens, float scale, int32_t num_splits,
                                  float *out_part, float *lse_part, int32_t flags,
                                  pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_decode_attn_noalloc -- the same computation as
 * pkv_paged_decode_attn (same arguments, same results), for callers that
 * cannot allocate device memory: the split partials go to a scratch array
 * built into the library instead of a caller workspace.  The pages have no
 * counterpart of this call; it exists for embedders whose host framework owns
 * all device memory, or whose hot loop must not allocate.
 *  - The scratch holds PKV_NOALLOC_SCRATCH_BYTES (8 MiB) on every GPU that
 *    loads the library, until the process exits.  A call whose partials
 *    (pkv_decode_workspace_size for the split count used) exceed it returns
 *    PKV_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 *  - The first call in each CUDA context looks up the scratch's device
 *    address; make that first call before any stream capture.
 *  - The request is checked as pkv_paged_decode_attn checks it (same
 *    statuses) before the scratch limit is applied.
 *  - Calls share the scratch: calls that overlap on the GPU race; calls in
 *    one stream are ordered.  Nothing is allocated, on host or device.
 * ------------------------------------------------------------------------- */
#define PKV_NOALLOC_SCRATCH_BYTES (8u << 20)

int pkv_paged_decode_attn_noalloc(const pkv_cache_desc *cache, const float *q, int32_t batch,
                                  int32_t num_q_heads, const void *k_pool, const void *v_pool,
                                  const int32_t *block_tables, int32_t max_blocks,
                                  const int32_t *seq_lens, float scale, int32_t num_splits,
                                  float *out, float *lse, int32_t flags, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_decode_attn_e4m3 -- pkv_paged_decode_attn over E4M3 pools (the
 * FP8 cache above): K_j = value(k code) * k_scale[g] and V_j = value(v code)
 * * v_scale[g]; q, out, lse, splits, workspace (pkv_decode_workspace_size)
 * and the status bits as pkv_paged_decode_attn; shapes as there.  Head
 * dims 128 with query groups of 4, 8, 16 or 32 (32 as two work items of 16
 * rows) and power-of-two block sizes 16..256 run on the tcgen05 tensor cores
 * with E4M3 operands: the fp32 query
 * is carried as four E4M3 terms and the probabilities as five, each term the
 * rounding residual of the one before scaled by 16, so both keep about 16
 * significant bits and the result is fp32-accurate attention on the stored
 * values.  Query groups that are a multiple of 64 heads (the MLA shape:
 * 128 heads over one 576-dim key / 512-dim value head; head dims multiples
 * of 64 / 128, power-of-two block sizes 64..256) run on the tcgen05
 * large-group kernel: each chunk's codes are expanded exactly into fp16 in
 * shared memory and the products run in fp16 with the query (scaled by a
 * power of two per work item) and the probabilities as fp16 hi + lo.
 * Other shapes, or flags PKV_DECODE_GENERIC / PKV_DECODE_NO_TCGEN05, run a
 * CUDA-core kernel that decodes the codes exactly.
 * ------------------------------------------------------------------------- */
/* The split count num_splits = 0 resolves to in pkv_paged_decode_attn_e4m3. */
int32_t pkv_decode_auto_splits_e4m3(const pkv_cache_desc *cache, int32_t batch,
                                    int32_t num_q_heads, int32_t max_seq_len);

int pkv_paged_decode_attn_e4m3(const pkv_cache_desc *cache, const float *q, int32_t batch,
                               int32_t num_q_heads, const void *k_pool, const void *v_pool,
                               const float *k_scale, const float *v_scale,
                               const int32_t *block_tables, int32_t max_blocks,
                               const int32_t *seq_lens, float scale, int32_t num_splits,
                               void *workspace, size_t workspace_bytes, float *out, float *lse,
                               int32_t flags, pkv_stream_t stream);

/* The per-chunk partials of pkv_paged_decode_attn_e4m3, as
 * pkv_paged_decode_attn_partial gives them for a bf16 cache: out_part
 * [S][batch][num_q_heads][head_dim_v] and lse_part [S][batch][num_q_heads]
 * (caller-owned device buffers, out_part 16-byte aligned), S = num_splits >= 1,
 * chunk s of row b covering [s*C_b, min(seq_lens[b], (s+1)*C_b)) with
 * C_b = 64 * ceil(seq_lens[b] / (64 * S)); an empty chunk gives out = 0 and
 * lse = -inf.  pkv_lse_merge of these equals pkv_paged_decode_attn_e4m3 at the
 * same S.  The [DCP] page's stage 3 merges such partials, one per
 * partition.  The test control flag is refused (PKV_ERR_INVALID_ARG). */
int pkv_paged_decode_attn_partial_e4m3(const pkv_cache_desc *cache, const float *q,
                                       int32_t batch, int32_t num_q_heads, const void *k_pool,
                                       const void *v_pool, const float *k_scale,
                                       const float *v_scale, const int32_t *block_tables,
                                       int32_t max_blocks, const int32_t *seq_lens, float scale,
                                       int32_t num_splits, float *out_part, float *lse_part,
                                       int32_t flags, pkv_stream_t stream);

/* pkv_paged_decode_attn_noalloc_e4m3 -- pkv_paged_decode_attn_e4m3 with the
 * split partials in the library's scratch (the rules of
 * pkv_paged_decode_attn_noalloc: PKV_NOALLOC_SCRATCH_BYTES, shared by all
 * calls, PKV_ERR_WORKSPACE_TOO_SMALL when the partials do not fit). */
int pkv_paged_decode_attn_noalloc_e4m3(const pkv_cache_desc *cache, const float *q,
                                       int32_t batch, int32_t num_q_heads, const void *k_pool,
                                       const void *v_pool, const float *k_scale,
                                       const float *v_scale, const int32_t *block_tables,
                                       int32_t max_blocks, const int32_t *seq_lens, float scale,
                                       int32_t num_splits, float *out, float *lse, int32_t flags,
                                       pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_decode_attn_multi -- several new tokens per sequence in one step
 * (e.g. verifying speculated tokens; [AX] names a speculative-verification
 * path among its decode kernels).  The last tokens_per_seq (T) of the
 * seq_lens[b] stored tokens of sequence b are the new ones, already appended;
 * query t (0-based) attends causally to the tokens j < seq_lens[b] - T + 1 + t:
 *     out[b][t][h][:], lse[b][t][h] = decode attention of q[b][t][h][:] over
 *     those tokens (the definition of pkv_paged_decode_attn).
 * q [batch][T][num_q_heads][head_dim_k], out [batch][T][num_q_heads][head_dim_v],
 * lse [batch][T][num_q_heads], fp32.  1 <= T <= 64.  A sequence holding fewer
 * than T tokens sets PKV_DEV_SEQ_LEN and its rows with no token give out = 0,
 * lse = -inf.  Splits, kernels and flags as for pkv_paged_decode_attn
 * (num_splits = 0: pkv_decode_multi_auto_splits).  When a GQA kernel takes
 * the shape with G * T rows per KV head (G = num_q_heads / num_kv_heads) --
 * the tcgen05 one at head dims 128 and G * T of 16 or 32 (32 as two work
 * items of 16 rows; not with PKV_DECODE_NO_TCGEN05), the TMA one at
 * G * T <= 16 -- the T tokens are extra rows of one work item and each K/V
 * tile is read once (twice from L2 at 32 rows); otherwise every (sequence, token) is attended as its own
 * row.  workspace: at least
 * pkv_decode_multi_workspace_size(...) bytes (never 0: it holds the T
 * per-token views of the block tables); contents on entry do not matter.
 * ------------------------------------------------------------------------- */
/* The split count num_splits = 0 resolves to for a multi-token call (same
 * arguments as that call's shape and flags) on the current device. */
int32_t pkv_decode_multi_auto_splits(const pkv_cache_desc *cache, int32_t batch,
                                     int32_t tokens_per_seq, int32_t num_q_heads,
                                     int32_t max_seq_len, int32_t flags);

size_t pkv_decode_multi_workspace_size(int32_t batch, int32_t tokens_per_seq,
                                       int32_t num_q_heads, int32_t head_dim_v,
                                       int32_t max_blocks, int32_t num_splits);

int pkv_paged_decode_attn_multi(const pkv_cache_desc *cache, const float *q, int32_t batch,
                                int32_t tokens_per_seq, int32_t num_q_heads, const void *k_pool,
                                const void *v_pool, const int32_t *block_tables,
                                int32_t max_blocks, const int32_t *seq_lens, float scale,
                                int32_t num_splits, void *workspace, size_t workspace_bytes,
                                float *out, float *lse, int32_t flags, pkv_stream_t stream);

/* pkv_paged_decode_attn_multi_e4m3 -- the multi-token step over E4M3 pools
 * (the FP8 cache above): rows, causal lengths, q/out/lse layouts, the
 * PKV_DEV_SEQ_LEN rule and the workspace (pkv_decode_multi_workspace_size)
 * as pkv_paged_decode_attn_multi; K_j, V_j, k_scale, v_scale and flags as
 * pkv_paged_decode_attn_e4m3.  With flags 0, head dims 128, power-of-two
 * block sizes 16..256 and G * T in {4, 8, 16, 32} (G = num_q_heads /
 * num_kv_heads; 32 as two work items of 16 rows), the tcgen05 E4M3 kernel takes the T tokens as rows of one
 * work item (causal limits per row) and each tile is read once; otherwise
 * every (sequence, token) is attended as its own row over a per-token view
 * of its table row.  num_splits = 0: pkv_decode_multi_auto_splits_e4m3. */
int32_t pkv_decode_multi_auto_splits_e4m3(const pkv_cache_desc *cache, int32_t batch,
                                          int32_t tokens_per_seq, int32_t num_q_heads,
                                          int32_t max_seq_len);

int pkv_paged_decode_attn_multi_e4m3(const pkv_cache_desc *cache, const float *q,
                                     int32_t batch, int32_t tokens_per_seq, int32_t num_q_heads,
                                     const void *k_pool, const void *v_pool,
                                     const float *k_scale, const float *v_scale,
                                     const int32_t *block_tables, int32_t max_blocks,
                                     const int32_t *seq_lens, float scale, int32_t num_splits,
                                     void *workspace, size_t workspace_bytes, float *out,
                                     float *lse, int32_t flags, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_decode_attn_cascade -- decode attention for sequences that share
 * a prefix.  [PA] "共通ブロックの共有とコピーオンライト": sequences with a common
 * prefix point their block tables at the same physical blocks; [AX]
 * "エージェントワークロードの特性": agent traffic re-sends long shared prefixes.
 * The result is pkv_paged_decode_attn's (same q, pools, tables, lengths,
 * scale, out and lse layouts) for tables whose first prefix_blocks entries
 * are prefix_table[0 .. prefix_blocks) (int32 device array), computed as a
 * cascade over the P = prefix_blocks * block_size shared tokens:
 *   1. every query row of every sequence attends to tokens [0, P) through
 *      prefix_table: the batch x num_q_heads rows form one sequence, so each
 *      staged prefix tile serves all the rows that need it (prefix_splits
 *      chunks);
 *   2. each sequence's rows attend to its own tokens [P, seq_lens[b])
 *      through the rest of its table row (suffix_splits chunks);
 *   3. the partials of 1 and 2 are merged as pkv_lse_merge merges.
 * A table that does not begin with prefix_table sets PKV_DEV_PREFIX (its
 * rows still use prefix_table for the first P tokens); seq_lens[b] < P sets
 * PKV_DEV_SEQ_LEN.  prefix_blocks may be 0 (no shared part) up to
 * max_blocks.  Split counts: 0 = chosen by pkv_decode_cascade_splits, else
 * 1..256.  workspace: at least pkv_decode_cascade_workspace_size(...) bytes,
 * 16-byte aligned; its contents on entry do not matter.  flags: 0, or
 * PKV_DECODE_GENERIC / PKV_DECODE_NO_TCGEN05 as for pkv_paged_decode_attn.
 * With flags 0 and query groups that are a multiple of 64 heads on the
 * tcgen05 kernel's head dims, both parts run in ONE launch of that kernel
 * (the suffix items fill the tail of the prefix items); otherwise as two
 * launches of whichever split kernel takes each part's shape.
 * ------------------------------------------------------------------------- */
/* Resolves zero split counts in *prefix_splits / *suffix_splits (others are
 * left as given) for the current device.  PKV_OK or PKV_ERR_INVALID_ARG. */
int pkv_decode_cascade_splits(const pkv_cache_desc *cache, int32_t batch, int32_t num_q_heads,
                              int32_t max_blocks, int32_t prefix_blocks,
                              int32_t *prefix_splits, int32_t *suffix_splits);

size_t pkv_decode_cascade_workspace_size(const pkv_cache_desc *cache, int32_t batch,
                                         int32_t num_q_heads, int32_t max_blocks,
                                         int32_t prefix_blocks, int32_t prefix_splits,
                                         int32_t suffix_splits);

int pkv_paged_decode_attn_cascade(const pkv_cache_desc *cache, const float *q, int32_t batch,
                                  int32_t num_q_heads, const void *k_pool, const void *v_pool,
                                  const int32_t *prefix_table, int32_t prefix_blocks,
                                  const int32_t *block_tables, int32_t max_blocks,
                                  const int32_t *seq_lens, float scale, int32_t prefix_splits,
                                  int32_t suffix_splits, void *workspace, size_t workspace_bytes,
                                  float *out, float *lse, int32_t flags, pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_lse_merge -- [DCP] decode step, stage 3: correct each partial output
 * with the shared LSEs and sum.  For each row r:
 *     M = max_p lse_part[p][r],  w_p = e^{lse_part[p][r] - M},
 *     out[r][:] = sum_p w_p out_part[p][r][:] / sum_p w_p,  lse[r] = M + ln sum_p w_p.
 * out_part [num_parts][rows][head_dim_v], lse_part [num_parts][rows],
 * out [rows][head_dim_v], lse [rows], all fp32.  Rows whose partials are all
 * empty (lse = -inf) give out = 0 and lse = -inf; a row with a NaN partial
 * LSE (an abandoned chunk) gives NaN.  out/lse must not alias the partials.
 * ------------------------------------------------------------------------- */
int pkv_lse_merge(int32_t num_parts, const float *out_part, const float *lse_part,
                  int64_t rows, int32_t head_dim_v, float *out, float *lse,
                  pkv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Host block manager -- [PA] "PagedAttentionはブロック表で論理順序と物理配置を分ける",
 * "要求の終了で空いたブロックを再利用する具体例", "共通ブロックの共有とコピーオンライト".
 * Host memory only; not thread-safe (one owner thread per manager).
 *  - A sequence uses its last block until it is full, then takes a free block.
 *  - Freed blocks return to the pool (last freed, first reused) and may be
 *    used by any sequence; nothing is compacted.
 *  - fork() makes a child that shares every block of its parent (each
 *    block's reference count goes up); a block returns to the pool only when
 *    its count reaches zero.
 *  - append() into a last block that other sequences still reference first
 *    takes a fresh block, reports (old, new) as a copy-on-write pair for
 *    pkv_copy_blocks, and points this sequence's table at the new block.
 *    Full shared blocks are never copied.
 * ------------------------------------------------------------------------- */
typedef struct pkv_block_manager pkv_block_manager;

/* `initial_order` (may be NULL = 0,1,2,...) is the order in which free blocks
 * are first handed out; it must be a permutation of 0..num_blocks-1. */
pkv_block_manager *pkv_bm_create(int32_t num_blocks, int32_t block_size,
                                 const int32_t *initial_order);
void pkv_bm_destroy(pkv_block_manager *bm);

/* New empty sequence; its id is written to *seq_id. */
int pkv_bm_add_sequence(pkv_block_manager *bm, int64_t *seq_id);

/* New sequence sharing all of `parent`'s blocks and length. */
int pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t *child);

/* Reserve slots for `num_tokens` new tokens of `seq`: slots_out[num_tokens]
 * receives their slots in order.  Copy-on-write pairs are written to
 * cow_src/cow_dst (capacity `cow_capacity`, at most 1 pair per call) and
 * their count to *num_cow.  All-or-nothing: PKV_ERR_NO_SPACE leaves the
 * manager unchanged. */
int pkv_bm_append(pkv_block_manager *bm, int64_t seq, int32_t num_tokens, int64_t *slots_out,
                  int32_t *cow_src, int32_t *cow_dst, int32_t cow_capacity, int32_t *num_cow);

/* Drop `seq`: every block's count goes down; blocks at zero return to the pool. */
int pkv_bm_free(pkv_block_manager *bm, int64_t seq);

/* Copy `seq`'s block table (logical order) into table_out[capacity]; the
 * number of blocks goes to *num_blocks and the token count to *seq_len. */
int pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq, int32_t *table_out,
                       int32_t capacity, int32_t *num_blocks, int64_t *seq_len);

int32_t pkv_bm_num_free(const pkv_block_manager *bm);
/* Reference count of a physical block (0 = free), or -1 if out of range. */
int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H_ */
