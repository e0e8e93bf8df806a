/*
 * oracle.c -- CPU oracle for paged decode attention over a block-table KV cache.
 *
 * TEST INFRASTRUCTURE.  This is the plain, slow statement of what the GPU
 * library computes.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the GPU library never calls it, and the two
 * share no code, header, helper or constant.  Every loop is written in the
 * order the method is described, in fp64, with no blocking or fusion.
 *
 * Pages this follows (cited by title and section):
 *   [PA]  "PagedAttentionとは？KVキャッシュを分割してLLMのメモリの無駄を減らす仕組み"
 *         sections "PagedAttentionはブロック表で論理順序と物理配置を分ける",
 *         "要求の終了で空いたブロックを再利用する具体例",
 *         "共通ブロックの共有とコピーオンライト".
 *   [KVB] "1,000 人が同時に AI に質問したら、誰が最初に答えをもらうのか? KV キャッシュと
 *         continuous batching", section "KV キャッシュは何を保持するのか?".
 *   [DCP] "なぜ長文LLMは遅くなるのか｜Decode Context ParallelismでKVキャッシュを分散する",
 *         the interleaved token assignment and the three-stage DCP decode step.
 *
 * Storage conventions (fixed by the tests that call this file, not by the pages):
 *   k_pool[num_blocks][num_kv_heads][block_size][head_dim_k]  bf16 bit patterns
 *   v_pool[num_blocks][num_kv_heads][block_size][head_dim_v]  bf16 bit patterns
 *   block_tables[B][max_blocks] int32, seq_lens[B] int32, q[B][Hq][Dk] fp32.
 *   Query head h reads KV head g = h / (Hq / Hkv)  (contiguous query groups).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* A bf16 value is the upper half of an IEEE binary32; widen it that way. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t wide = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &wide, sizeof f);
    return (double)f;
}

/* FP8 storage of the cache.  [DCP] counts a cached number's bytes by data
 * type (FP8: one byte) and describes KV-cache quantisation as storing the
 * cache in a low-precision type such as FP8 so that each token takes fewer
 * bytes; [PA] "Continuous Batching・prefix caching・量子化との違い": quantisation
 * changes the stored representation, so its effect on accuracy has to be
 * checked.  The pages fix no format; this oracle reads "FP8" as E4M3: one
 * sign bit, four exponent bits with bias 7, three mantissa bits; exponent
 * field 0 holds the subnormals m/8 * 2^-6; there are no infinities and
 * S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* The E4M3 code nearest to x, a tie going to the even mantissa; magnitudes
 * of 448 and beyond (infinities too) give +-448, NaN gives NaN. */
uint8_t oracle_e4m3_from_double(double x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {
        /* subnormal binade, steps of 2^-9; 8 steps is 2^-6, whose code is 8 */
        double m = nearbyint(a / ldexp(1.0, -9));
        return sign | (uint8_t)m;
    }
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                       /* a in [2^e, 2^(e+1)) */
    double m = nearbyint((a / ldexp(1.0, e) - 1.0) * 8.0);
    if (m == 8.0) {
        m = 0.0;
        e += 1;
    }
    int code = ((e + 7) << 3) | (int)m;
    if (code > 0x7e)
        code = 0x7e;
    return sign | (uint8_t)code;
}

/* [PA] "PagedAttentionはブロック表で論理順序と物理配置を分ける": the block table maps the
 * n-th logical block of a sequence to the physical block that stores it, so
 * logical token `pos` lives in physical block table_row[pos / bs] at offset
 * pos % bs. */
int64_t oracle_slot_of(const int32_t *table_row, int64_t pos, int32_t block_size)
{
    int64_t logical_block = pos / block_size;
    int64_t offset = pos % block_size;
    return (int64_t)table_row[logical_block] * block_size + offset;
}

/* [KVB] "KV キャッシュは何を保持するのか?": a decode step computes the new token's key
 * and value and adds them to the cache.  Token t is written at slot
 * slot_mapping[t]; a negative slot means "no token" and is skipped.  Returns
 * the number of slots that were out of range (those are skipped too). */
int64_t oracle_kv_append(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim_k, int32_t head_dim_v,
                         uint16_t *k_pool, uint16_t *v_pool,
                         const uint16_t *k_new, const uint16_t *v_new,
                         const int64_t *slot_mapping, int64_t num_tokens)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            ++bad;
            continue;
        }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            for (int32_t d = 0; d < head_dim_k; ++d)
                k_pool[((block * num_kv_heads + g) * block_size + offset) * head_dim_k + d] =
                    k_new[(t * num_kv_heads + g) * head_dim_k + d];
            for (int32_t d = 0; d < head_dim_v; ++d)
                v_pool[((block * num_kv_heads + g) * block_size + offset) * head_dim_v + d] =
                    v_new[(t * num_kv_heads + g) * head_dim_v + d];
        }
    }
    return bad;
}

/* The same scatter into E4M3 pools (uint8).  Element x (bf16) of KV head g
 * is stored as the code nearest to x / s_g, the quotient taken in binary32
 * (correctly rounded), where s_g = k_scale[g] or v_scale[g] is that head's
 * dequantisation scale: the stored element reads back as decode * s_g. */
int64_t oracle_kv_append_e4m3(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                              int32_t head_dim_k, int32_t head_dim_v,
                              uint8_t *k_pool, uint8_t *v_pool,
                              const uint16_t *k_new, const uint16_t *v_new,
                              const float *k_scale, const float *v_scale,
                              const int64_t *slot_mapping, int64_t num_tokens)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            ++bad;
            continue;
        }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            for (int32_t d = 0; d < head_dim_k; ++d) {
                float x = (float)oracle_bf16_to_double(k_new[(t * num_kv_heads + g) * head_dim_k + d]);
                float y = x / k_scale[g];
                k_pool[((block * num_kv_heads + g) * block_size + offset) * head_dim_k + d] =
                    oracle_e4m3_from_double((double)y);
            }
            for (int32_t d = 0; d < head_dim_v; ++d) {
                float x = (float)oracle_bf16_to_double(v_new[(t * num_kv_heads + g) * head_dim_v + d]);
                float y = x / v_scale[g];
                v_pool[((block * num_kv_heads + g) * block_size + offset) * head_dim_v + d] =
                    oracle_e4m3_from_double((double)y);
            }
        }
    }
    return bad;
}

/* [PA] "共通ブロックの共有とコピーオンライト": before a sequence writes into a block it
 * shares, the block is duplicated and that sequence's table is pointed at the
 * copy.  This is the duplication: every KV head's K and V rows of block src[i]
 * are copied to block dst[i].  Returns the number of pairs skipped because a
 * block id was out of range. */
int32_t oracle_copy_blocks(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                           int32_t head_dim_k, int32_t head_dim_v,
                           uint16_t *k_pool, uint16_t *v_pool,
                           const int32_t *src, const int32_t *dst, int32_t num_pairs)
{
    int32_t bad = 0;
    size_t k_block = (size_t)num_kv_heads * block_size * head_dim_k;
    size_t v_block = (size_t)num_kv_heads * block_size * head_dim_v;
    for (int32_t i = 0; i < num_pairs; ++i) {
        if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) {
            ++bad;
            continue;
        }
        memcpy(k_pool + (size_t)dst[i] * k_block, k_pool + (size_t)src[i] * k_block,
               k_block * sizeof(uint16_t));
        memcpy(v_pool + (size_t)dst[i] * v_block, v_pool + (size_t)src[i] * v_block,
               v_block * sizeof(uint16_t));
    }
    return bad;
}

/* [DCP] interleaved assignment: with interleave size I and P partitions, the
 * KV of token i belongs to partition (i / I) mod P, and each partition keeps
 * its tokens in their original relative order.  part[i] receives the
 * partition and local[i] the position of token i inside that partition,
 * found by counting the tokens already given to the partition. */
void oracle_interleave(int64_t num_tokens, int32_t num_parts, int32_t interleave,
                       int32_t *part, int64_t *local)
{
    int64_t *count = calloc((size_t)num_parts, sizeof(int64_t));
    for (int64_t i = 0; i < num_tokens; ++i) {
        int32_t r = (int32_t)((i / interleave) % num_parts);
        part[i] = r;
        local[i] = count[r];
        count[r] += 1;
    }
    free(count);
}

/* [DCP] three-stage decode step, stage 3: the partial outputs are corrected
 * with the shared log-sum-exp values and then summed.  Written out: with
 * M = max_p lse_p and w_p = exp(lse_p - M),
 *     out = sum_p w_p * out_p / sum_p w_p,     lse = M + log(sum_p w_p).
 * A row whose partials are all empty (lse = -inf) stays empty: out = 0,
 * lse = -inf.  Layout: out_part[P][rows][dv], lse_part[P][rows]. */
void oracle_lse_merge(int32_t num_parts, int64_t rows, int32_t head_dim_v,
                      const double *out_part, const double *lse_part,
                      double *out, double *lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int32_t p = 0; p < num_parts; ++p)
            if (lse_part[p * rows + r] > m)
                m = lse_part[p * rows + r];
        if (m == -INFINITY) {
            for (int32_t d = 0; d < head_dim_v; ++d)
                out[r * head_dim_v + d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int32_t p = 0; p < num_parts; ++p)
            wsum += exp(lse_part[p * rows + r] - m);
        for (int32_t d = 0; d < head_dim_v; ++d) {
            double acc = 0.0;
            for (int32_t p = 0; p < num_parts; ++p) {
                double w = exp(lse_part[p * rows + r] - m);
                acc += w * out_part[(p * rows + r) * head_dim_v + d];
            }
            out[r * head_dim_v + d] = acc / wsum;
        }
        lse[r] = m + log(wsum);
    }
}

/* ---------------------------------------------------------------------------
 * Decode attention of one new query token per sequence.
 *
 * [PA] "PagedAttentionはブロック表で論理順序と物理配置を分ける": attention reads the
 * scattered KV through the block table; the logical order and the context it
 * refers to are unchanged, so the result is exact softmax attention over the
 * tokens in logical order.  [KVB] "KV キャッシュは何を保持するのか?": the new token's
 * query is compared with the keys of all earlier tokens and the result weights
 * their values.  [DCP] requires the log-sum-exp of the softmax as a second
 * output; it is the natural log of sum_j exp(s_j) of the scaled scores s_j.
 *
 * For row (b, h), with g = h / (Hq / Hkv), over tokens j in [begin_b, end_b):
 *     s_j  = scale * sum_d q[b][h][d] * K_j[d]
 *     M    = max_j s_j,  Z = sum_j exp(s_j - M)
 *     out  = sum_j exp(s_j - M) * V_j / Z,   lse = M + log Z
 * An empty range gives out = 0 and lse = -inf.  begin/end default to
 * [0, seq_lens[b]) when the pointers are NULL.  K_j and V_j are the cached
 * numbers: bf16 values, or for E4M3 pools decode(code) * s_g.
 * ------------------------------------------------------------------------- */
typedef struct {
    int32_t B, Hq, Hkv, Dk, Dv, bs, max_blocks;
    const float *q;
    const uint16_t *k_pool, *v_pool;     /* bf16 pools, or NULL */
    const uint8_t *k8, *v8;              /* E4M3 pools, or NULL */
    const float *k_scale, *v_scale;      /* E4M3 dequantisation scales per KV head */
    const int32_t *block_tables, *seq_lens, *tok_begin, *tok_end;
    double scale;
    double *out, *lse;
    int64_t row_first, row_step;
} attn_job;

static double k_elem(const attn_job *J, int64_t idx, int32_t g)
{
    return J->k8 ? oracle_e4m3_to_double(J->k8[idx]) * J->k_scale[g]
                 : oracle_bf16_to_double(J->k_pool[idx]);
}

static double v_elem(const attn_job *J, int64_t idx, int32_t g)
{
    return J->v8 ? oracle_e4m3_to_double(J->v8[idx]) * J->v_scale[g]
                 : oracle_bf16_to_double(J->v_pool[idx]);
}

static void attend_row(const attn_job *J, int64_t row, double *scores)
{
    int32_t b = (int32_t)(row / J->Hq);
    int32_t h = (int32_t)(row % J->Hq);
    int32_t g = h / (J->Hq / J->Hkv);
    int64_t begin = J->tok_begin ? J->tok_begin[b] : 0;
    int64_t end = J->tok_end ? J->tok_end[b] : J->seq_lens[b];
    if (end > J->seq_lens[b])
        end = J->seq_lens[b];
    double *o = J->out + row * J->Dv;
    for (int32_t d = 0; d < J->Dv; ++d)
        o[d] = 0.0;
    if (begin >= end) {
        J->lse[row] = -INFINITY;
        return;
    }
    const float *qrow = J->q + row * J->Dk;
    const int32_t *table_row = J->block_tables + (int64_t)b * J->max_blocks;

    double m = -INFINITY;
    for (int64_t j = begin; j < end; ++j) {
        int64_t phys = table_row[j / J->bs];
        int64_t off = j % J->bs;
        int64_t krow = ((phys * J->Hkv + g) * J->bs + off) * J->Dk;
        double dot = 0.0;
        for (int32_t d = 0; d < J->Dk; ++d)
            dot += (double)qrow[d] * k_elem(J, krow + d, g);
        scores[j - begin] = J->scale * dot;
        if (scores[j - begin] > m)
            m = scores[j - begin];
    }
    double z = 0.0;
    for (int64_t j = begin; j < end; ++j) {
        double p = exp(scores[j - begin] - m);
        z += p;
        int64_t phys = table_row[j / J->bs];
        int64_t off = j % J->bs;
        int64_t vrow = ((phys * J->Hkv + g) * J->bs + off) * J->Dv;
        for (int32_t d = 0; d < J->Dv; ++d)
            o[d] += p * v_elem(J, vrow + d, g);
    }
    for (int32_t d = 0; d < J->Dv; ++d)
        o[d] /= z;
    J->lse[row] = m + log(z);
}

static void *attend_rows(void *arg)
{
    const attn_job *J = (const attn_job *)arg;
    int64_t rows = (int64_t)J->B * J->Hq;
    int64_t longest = 1;
    for (int32_t b = 0; b < J->B; ++b)
        if (J->seq_lens[b] > longest)
            longest = J->seq_lens[b];
    double *scores = malloc((size_t)longest * sizeof(double));
    for (int64_t row = J->row_first; row < rows; row += J->row_step)
        attend_row(J, row, scores);
    free(scores);
    return NULL;
}

/* Runs `proto` (row_first/row_step ignored) over all rows: `num_threads` <= 0
 * uses every online core; rows are dealt out round-robin, which changes no
 * arithmetic (each row is computed by exactly one thread, in the order above). */
static int32_t run_attn(attn_job proto, int32_t num_threads)
{
    const int32_t B = proto.B, Hq = proto.Hq, Hkv = proto.Hkv, block_size = proto.bs;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || block_size <= 0)
        return -1;
    if (num_threads <= 0)
        num_threads = (int32_t)sysconf(_SC_NPROCESSORS_ONLN);
    if (num_threads < 1)
        num_threads = 1;
    int64_t rows = (int64_t)B * Hq;
    if (num_threads > rows)
        num_threads = (int32_t)(rows > 0 ? rows : 1);
    attn_job *jobs = malloc(sizeof(attn_job) * (size_t)num_threads);
    pthread_t *tids = malloc(sizeof(pthread_t) * (size_t)num_threads);
    for (int32_t t = 0; t < num_threads; ++t) {
        jobs[t] = proto;
        jobs[t].row_first = t;
        jobs[t].row_step = num_threads;
    }
    if (num_threads == 1) {
        attend_rows(&jobs[0]);
    } else {
        for (int32_t t = 0; t < num_threads; ++t)
            pthread_create(&tids[t], NULL, attend_rows, &jobs[t]);
        for (int32_t t = 0; t < num_threads; ++t)
            pthread_join(tids[t], NULL);
    }
    free(jobs);
    free(tids);
    return 0;
}

/* Returns 0, or -1 if the arguments are inconsistent. */
int32_t oracle_paged_decode_attn(int32_t B, int32_t Hq, int32_t Hkv, int32_t Dk, int32_t Dv,
                                 int32_t block_size, int32_t max_blocks, const float *q,
                                 const uint16_t *k_pool, const uint16_t *v_pool,
                                 const int32_t *block_tables, const int32_t *seq_lens,
                                 const int32_t *tok_begin, const int32_t *tok_end,
                                 double scale, double *out, double *lse, int32_t num_threads)
{
    attn_job J = {B, Hq, Hkv, Dk, Dv, block_size, max_blocks, q, k_pool, v_pool,
                  NULL, NULL, NULL, NULL, block_tables, seq_lens, tok_begin, tok_end,
                  scale, out, lse, 0, 1};
    return run_attn(J, num_threads);
}

/* The same over E4M3 pools with per-KV-head dequantisation scales. */
int32_t oracle_paged_decode_attn_e4m3(int32_t B, int32_t Hq, int32_t Hkv, int32_t Dk, int32_t Dv,
                                      int32_t block_size, int32_t max_blocks, const float *q,
                                      const uint8_t *k_pool, const uint8_t *v_pool,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_tables, const int32_t *seq_lens,
                                      const int32_t *tok_begin, const int32_t *tok_end,
                                      double scale, double *out, double *lse,
                                      int32_t num_threads)
{
    attn_job J = {B, Hq, Hkv, Dk, Dv, block_size, max_blocks, q, NULL, NULL,
                  k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, tok_begin,
                  tok_end, scale, out, lse, 0, 1};
    return run_attn(J, num_threads);
}
