// decode_gqa_tc.cu -- paged decode attention for 16 query rows per KV head
// (a 16-head query group, or 4 heads x 4 new tokens of a multi-token step)
// with head dims 128, on the 5th-generation tensor cores of sm_103a.
//
// At 16 rows the warp-level-MMA GQA kernel is bound by its own MMAs (the
// fp32 query and probabilities go through bf16 as hi + lo pairs: four times
// the MMAs per byte of a 4-head group); here the same products run as
// tcgen05 MMAs with fp32 accumulators in tensor memory, and the CUDA cores
// only do the softmax.
//
// Work item = (sequence b, KV head g, split chunk s), walked in 128-token
// tiles:
//   S^T[128 tok x 32] = K_tile . [Q_hi ; Q_lo]^T    (M=128, N=32: the 16 rows'
//                                                    hi and lo halves stacked)
//   online softmax over the 128 token lanes            (CUDA cores)
//   O^T[128 dv x 32] += V_tile^T . [P_hi ; P_lo]^T    (M=128, N=32)
// so one MMA per 16-element k-step covers both halves; the epilogue adds the
// hi and lo columns of S^T and of O^T.  TMEM: two 32-column S^T buffers and
// the 32-column O^T (128 columns allocated); shared memory ~92 KB, so two
// CTAs share an SM and keep eight 16 KB stages of K/V in flight.
//
// A ring stage holds 64 tokens x 128 dims as [8-token group][64-dim half]
// [8 rows][128 B] (128-byte swizzle): each TMA box is one KV block (at most
// 64 tokens) of whole 256-byte rows, so a block is fetched as one contiguous
// run.  A K tile is two adjacent stages read by every score MMA (8-row atoms
// 2048 B apart, the second half of the dims at +1024); a V stage is the value
// MMAs' MN-major operand for 64 tokens (halves 1024 B apart, token groups
// 2048 B apart).
//
// Warp roles (192 threads): warp 0 issues the TMA copies (lane j loads box
// j, blocks of 16..256 tokens); warp 1 owns the TMEM allocation, issues
// every MMA from one thread and zeroes value rows past a sequence's end;
// warps 2-5 are one thread per TMEM lane (token row of S^T, value row of O^T)
// for the query split, the softmax and the epilogue.  A row's running max is
// raised only when a score exceeds it by more than 8 (log2 units); then the
// accumulators are rescaled in TMEM.  Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_math.cuh"
#include "pkv_host.h"
#include "pkv_pipeline.cuh"
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kRows = 16;               // query rows per work item
constexpr int kN = 2 * kRows;           // MMA N: hi rows | lo rows
constexpr int kM = 128;                 // tokens per tile
constexpr int kD = 128;                 // head dim (K and V)
constexpr int kChunk = 16384;           // bytes per ring stage
#ifndef PKV_GQA_TC_RING
#define PKV_GQA_TC_RING 4
#endif
#ifndef PKV_GQA_TC_CTAS
#define PKV_GQA_TC_CTAS 2
#endif
constexpr int kRing = PKV_GQA_TC_RING;  // ring stages per CTA
constexpr int kCtas = PKV_GQA_TC_CTAS;  // CTAs per SM
constexpr int kThreads = 192;
constexpr int kSoftWarp0 = 2;
constexpr int kSoftThreads = 128;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColS = 0;           // S^T buffers at columns 0 and 32
constexpr uint32_t kColO = 64;          // O^T at columns 64..95
constexpr float kSlack = 8.f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kIdS = tc::idesc_bf16_f32(128, kN, 0, 0);   // K-major K, K-major Q
constexpr uint32_t kIdO = tc::idesc_bf16_f32(128, kN, 1, 0);   // MN-major V, K-major P

// mbarrier slots
constexpr int kBarFull = 0;             // + stage (up to 12)
constexpr int kBarEmpty = 12;           // + stage
constexpr int kBarSFull = 24;           // + buffer
constexpr int kBarSEmpty = 26;          // + buffer
constexpr int kBarPFull = 28;           // + P buffer: probabilities written (128 arrivals)
constexpr int kBarPvDone = 30;          // + P buffer: value MMAs reading it done (commit)
constexpr int kBarQFull = 32;
constexpr int kBarQEmpty = 33;
constexpr int kBarOEmpty = 34;
constexpr int kBarDrain = 35;
static_assert(PKV_GQA_TC_RING <= 12, "mbarrier slots for at most 12 stages");
static_assert(PKV_GQA_TC_RING % 2 == 0, "a K tile takes two adjacent stages");

// Shared memory, offsets from a 1024-byte-aligned base.
constexpr uint32_t kOffBars = 0;
constexpr uint32_t kOffMrow = 48 * 8;                  // running max per row (log2)
constexpr uint32_t kOffAux = kOffMrow + kRows * 4;     // rescale factor / 1 / l
constexpr uint32_t kOffRed = kOffAux + kRows * 4;      // [4 warps][16 rows]
constexpr uint32_t kOffSlot = kOffRed + 4 * kRows * 4;
constexpr uint32_t kOffFlag = kOffSlot + 4;
constexpr uint32_t kOffQ = 1024;                       // [2 segs][32 rows][128 B]
constexpr uint32_t kPBytes = 2 * kN * 128;             // [2 token atoms][32 rows][128 B]
constexpr uint32_t kOffP = kOffQ + 2 * kN * 128;       // two P buffers (tile parity)
constexpr uint32_t kOffRing = kOffP + 2 * kPBytes;
constexpr uint32_t kSmemBytes = 1024 + kOffRing + kRing * kChunk;

__device__ __forceinline__ int64_t lmin(int64_t x, int64_t y) { return x < y ? x : y; }

struct Item {
    int b, g, s, hg;
    int64_t len, begin, end;
    int ntiles;
};

// Head groups per (sequence, KV head): the item's 16 rows are 16 / T heads x
// T query tokens, so G x T = 32 rows are two items.
__device__ __forceinline__ int head_groups(const DecodeArgs &a) {
    return a.num_q_heads / a.cache.num_kv_heads * a.q_tokens / kRows;
}

// item = ((b * Hkv + g) * S + s) * HG + hg: the head groups of one
// (sequence, KV head, split) are neighbours and read the same tiles together.
__device__ __forceinline__ Item gqa_item(const DecodeArgs &a, int item, bool report) {
    Item r;
    const int HG = head_groups(a);
    r.hg = item % HG;
    const int t0 = item / HG;
    r.s = t0 % a.num_splits;
    const int t = t0 / a.num_splits;
    r.g = t % a.cache.num_kv_heads;
    r.b = t / a.cache.num_kv_heads;
    int64_t L = a.seq_lens[r.b];
    report = report && r.s == 0 && r.hg == 0;
    if (L < 0 || L > int64_t(a.max_blocks) * a.cache.block_size) {
        if (report) raise_status(a.status, PKV_DEV_SEQ_LEN);
        L = 0;
    } else if (L < a.flag_below && report) {
        raise_status(a.status, PKV_DEV_SEQ_LEN);
    }
    const int64_t chunk = 64 * ((L + 64LL * a.num_splits - 1) / (64LL * a.num_splits));
    r.len = L;
    r.begin = int64_t(r.s) * chunk;
    r.end = lmin(L, r.begin + chunk);
    r.ntiles = r.end > r.begin ? int((r.end - r.begin + kM - 1) / kM) : 0;
    return r;
}

// Row `row` of an item -> its query / output row, in head vectors: query
// token t = row / Gr of sequence b, head g G + hg Gr + row % Gr.
__device__ __forceinline__ int64_t row_offset(const DecodeArgs &a, const Item &r, int row, int Gr) {
    const int t = row / Gr, h = row - t * Gr;
    const int G = a.num_q_heads / a.cache.num_kv_heads;
    return (int64_t(r.b) * a.q_tokens + t) * a.num_q_heads + int64_t(r.g) * G + r.hg * Gr + h;
}

// Offset of bf16 element (row, col < 64) in a [rows][64] 128-byte-swizzled
// array whose 8-row atoms are 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t(row) * 128 + (uint32_t(((col >> 3) ^ row) & 7) << 4) + uint32_t(col & 7) * 2;
}

__global__ void __launch_bounds__(kThreads, kCtas)
decode_gqa_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(base);
    float *mrow = reinterpret_cast<float *>(base + kOffMrow);
    float *aux = reinterpret_cast<float *>(base + kOffAux);
    float *red = reinterpret_cast<float *>(base + kOffRed);
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(base + kOffSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kOffFlag);
    auto bar = [&](int i) { return sb + kOffBars + 8u * uint32_t(i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_items = a.batch * a.cache.num_kv_heads * a.num_splits * head_groups(a);
    const int bs = a.cache.block_size, hkv = a.cache.num_kv_heads;
    const int box = bs < 64 ? bs : 64;                  // rows per TMA box (one block or less)
    const int T = a.q_tokens, Gr = kRows / a.q_tokens;   // query tokens, heads per item

    if (threadIdx.x == 0) {
        for (int r = 0; r < kRing; ++r) {
            mbar_init(bar(kBarFull + r), 1);
            mbar_init(bar(kBarEmpty + r), 1);
        }
        mbar_init(bar(kBarSFull), 1);
        mbar_init(bar(kBarSFull + 1), 1);
        mbar_init(bar(kBarSEmpty), kSoftThreads);
        mbar_init(bar(kBarSEmpty + 1), kSoftThreads);
        mbar_init(bar(kBarPFull), kSoftThreads);
        mbar_init(bar(kBarPFull + 1), kSoftThreads);
        mbar_init(bar(kBarPvDone), 1);
        mbar_init(bar(kBarPvDone + 1), 1);
        mbar_init(bar(kBarQFull), kSoftThreads);
        mbar_init(bar(kBarQEmpty), 1);
        mbar_init(bar(kBarOEmpty), kSoftThreads);
        mbar_init(bar(kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::alloc(sb + kOffSlot, kTmemCols);
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // -------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        int stage = 0;
        uint32_t phase = 0, armed = 0, armed_parity = 0;
        bool ok = true;
        auto acquire = [&](uint32_t &dst) -> bool {
            const bool w = pipe_wait(bar(kBarEmpty + stage), phase ^ 1u, a.status, abort_flag);
            if (!__all_sync(0xffffffffu, w)) return false;
            if (lane == 0) mbar_arrive_expect_tx(bar(kBarFull + stage), kChunk);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            dst = sb + kOffRing + uint32_t(stage) * kChunk;
            return true;
        };
        auto advance = [&]() {
            if (++stage == kRing) {
                stage = 0;
                phase ^= 1u;
            }
        };
        const int nbox = kM / box;                     // boxes per 128-token tile (<= 8)
        const int per_stage = 64 / box;                // boxes per 64-token stage
        for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
            const Item r = gqa_item(a, item, false);
            if (r.ntiles == 0) continue;
            const int32_t *table = a.block_tables + int64_t(r.b) * a.max_blocks;
            // Rows of block 0 of this KV head stand in for boxes past the end
            // (masked scores, zeroed value rows).
            const int32_t standin = r.g * bs;
            int32_t yprev = standin;
            for (int i = 0; i <= r.ntiles && ok; ++i) {
                // lane j < nbox: global row of box j of tile i
                int32_t y = standin;
                if (i < r.ntiles && lane < nbox) {
                    const int64_t t = r.begin + int64_t(i) * kM + int64_t(lane) * box;
                    if (t < r.end) {
                        const int32_t phys = table[t / bs];
                        if (phys >= 0 && phys < a.cache.num_blocks)
                            y = (phys * hkv + r.g) * bs + int32_t(t % bs);
                        else
                            raise_status(a.status, PKV_DEV_BLOCK_ID);
                    }
                }
                // stage h of a tile: tokens 64h..64h+63; lane j issues box j
                // (after lane 0 armed the stage), box j - h * per_stage of it
                for (int kv = (i < r.ntiles ? 0 : 1); kv < (i > 0 ? 2 : 1) && ok; ++kv) {
                    const CUtensorMap *map = kv == 0 ? &tmap_k : &tmap_v;   // K(i), V(i-1)
                    const int32_t yb = kv == 0 ? y : yprev;
                    for (int h = 0; h < 2; ++h) {
                        uint32_t dst;
                        if (!acquire(dst)) {
                            ok = false;
                            break;
                        }
                        const int j = lane - h * per_stage;
                        __syncwarp();
                        if (j >= 0 && j < per_stage)
                            tma_load_4d(dst + uint32_t(j * box) * 256, map, 0, 0, 0, yb >> 3,
                                        bar(kBarFull + stage));
                        advance();
                    }
                }
                yprev = y;
            }
        }
        if (lane == 0)
            for (int s = 0; s < kRing; ++s)
                if (armed & (1u << s))
                    mbar_wait(bar(kBarFull + s), (armed_parity >> s) & 1u, a.status);
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        int stage = 0;
        uint32_t phase = 0, tcount = 0, pcount = 0, ne = 0;
        bool ok = true;
        const uint32_t qb = sb + kOffQ, pb = sb + kOffP;
        auto wait_all = [&](uint32_t b, uint32_t parity) {
            return __all_sync(0xffffffffu, pipe_wait(b, parity, a.status, abort_flag));
        };
        auto advance = [&]() {
            if (++stage == kRing) {
                stage = 0;
                phase ^= 1u;
            }
        };
        for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
            const Item r = gqa_item(a, item, false);
            if (r.ntiles == 0) continue;
            if (!(ok = wait_all(bar(kBarQFull), ne & 1u))) break;
            for (int i = 0; i <= r.ntiles && ok; ++i) {
                if (i < r.ntiles) {
                    const uint32_t buf = tcount & 1u;
                    if (!(ok = wait_all(bar(kBarSEmpty + buf), ((tcount >> 1) & 1u) ^ 1u))) break;
                    const uint32_t d = tmem + kColS + kN * buf;
                    // both stages of the tile (stage is even: they are adjacent)
                    if (!(ok = wait_all(bar(kBarFull + stage), phase) &&
                               wait_all(bar(kBarFull + stage + 1), phase)))
                        break;
                    tc::fence_after_sync();
                    if (lane == 0) {
                        const uint32_t kb = sb + kOffRing + uint32_t(stage) * kChunk;
#pragma unroll
                        for (int seg = 0; seg < 2; ++seg)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc::mma_bf16(d, tc::smem_desc(kb + seg * 1024 + 32 * kk, 16, 2048),
                                             tc::smem_desc(qb + seg * kN * 128 + 32 * kk, 16, 1024),
                                             kIdS, (seg | kk) != 0);
                        tc::commit(bar(kBarEmpty + stage));
                        tc::commit(bar(kBarEmpty + stage + 1));
                    }
                    __syncwarp();
                    advance();
                    advance();
                    if (lane == 0) {
                        tc::commit(bar(kBarSFull + buf));
                        if (i == r.ntiles - 1) tc::commit(bar(kBarQEmpty));
                    }
                    __syncwarp();
                    ++tcount;
                }
                if (i > 0) {
                    // global value tile pcount reads P buffer pcount & 1
                    const int j = i - 1;
                    const uint32_t pbuf = pcount & 1u;
                    if (!(ok = wait_all(bar(kBarPFull + pbuf), (pcount >> 1) & 1u))) break;
                    if (j == 0 && !(ok = wait_all(bar(kBarOEmpty), (ne & 1u) ^ 1u))) break;
                    const int64_t tok0 = r.begin + int64_t(j) * kM;
                    const int nvalid = int(lmin(kM, r.end - tok0));
                    for (int h = 0; h < 2; ++h) {
                        if (!(ok = wait_all(bar(kBarFull + stage), phase))) break;
                        const int first_bad = nvalid - h * 64;
                        if (first_bad < 64) {
                            uint8_t *vt = base + kOffRing + size_t(stage) * kChunk;
                            const int r0 = first_bad > 0 ? first_bad : 0;
                            for (int idx = lane; idx < (64 - r0) * 16; idx += 32) {
                                const int row = r0 + (idx >> 4), c = idx & 15;
                                *reinterpret_cast<uint4 *>(vt + (row >> 3) * 2048 + (c >> 3) * 1024 +
                                                           (row & 7) * 128 + (c & 7) * 16) =
                                    make_uint4(0, 0, 0, 0);
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                        }
                        tc::fence_after_sync();
                        if (lane == 0) {
                            const uint32_t vb = sb + kOffRing + uint32_t(stage) * kChunk;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc::mma_bf16(tmem + kColO,
                                             tc::smem_desc(vb + 4096 * kk, 1024, 2048),
                                             tc::smem_desc(pb + pbuf * kPBytes + h * kN * 128 +
                                                               32 * kk, 16, 1024),
                                             kIdO, (j | h | kk) != 0);
                            tc::commit(bar(kBarEmpty + stage));
                        }
                        __syncwarp();
                        advance();
                    }
                    if (!ok) break;
                    if (lane == 0) tc::commit(bar(kBarPvDone + pbuf));
                    __syncwarp();
                    ++pcount;
                }
            }
            ++ne;
        }
        if (lane == 0) {
            tc::commit(bar(kBarDrain));
            mbar_wait(bar(kBarDrain), 0, a.status);
        }
        __syncwarp();
    } else {
        // -------------------------------------------- softmax and epilogue
        const int t = threadIdx.x - kSoftWarp0 * 32;     // 0..127
        const int quad = warp & 3;
        const int row = quad * 32 + lane;                // token row / value row
        const uint32_t tl = tmem + (uint32_t(quad * 32) << 16);
        const float qscale = a.scale * kLog2e;
        uint8_t *qs = base + kOffQ, *ps = base + kOffP;
        uint32_t tcount = 0, pcount = 0, ne = 0;   // pcount: probability tiles written
        // Wait until the value MMAs of global tile j (which read P buffer
        // j & 1) are done; waiting twice for one tile is harmless (the
        // buffer's next phase needs probabilities not yet written).
        auto wait_pv = [&](uint32_t j) {
            return pipe_wait(bar(kBarPvDone + (j & 1u)), (j >> 1) & 1u, a.status, abort_flag);
        };
        // The item's 16 query rows, pre-scaled, as bf16 hi (rows 0-15) and
        // lo (rows 16-31) of the score MMA's B operand, once the previous
        // item's score MMAs are done (completion `qphase` of QEmpty).
        auto stage_q = [&](const Item &q_item, uint32_t qphase) {
            const bool ok_q =
                pipe_wait(bar(kBarQEmpty), (qphase & 1u) ^ 1u, a.status, abort_flag);
            if (ok_q) {
                for (int i = t; i < kRows * kD / 2; i += kSoftThreads) {
                    const int rr = i / (kD / 2), d = 2 * (i % (kD / 2));
                    const float2 x = *reinterpret_cast<const float2 *>(
                        a.q + row_offset(a, q_item, rr, Gr) * kD + d);
                    const float x0 = x.x * qscale, x1 = x.y * qscale;
                    const uint32_t hi = pack_bf16x2(x0, x1);
                    const uint32_t lo =
                        pack_bf16x2(x0 - bf16_lo_to_f32(hi), x1 - bf16_hi_to_f32(hi));
                    const uint32_t seg = uint32_t(d >> 6) * kN * 128;
                    *reinterpret_cast<uint32_t *>(qs + seg + swz(rr, d & 63)) = hi;
                    *reinterpret_cast<uint32_t *>(qs + seg + swz(kRows + rr, d & 63)) = lo;
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(bar(kBarQFull));
            return ok_q;
        };
        // The next item after `from` that has tokens (-1: none).
        auto next_busy = [&](int from, Item &nx) {
            for (int it = from + gridDim.x; it < num_items; it += gridDim.x) {
                nx = gqa_item(a, it, false);
                if (nx.ntiles > 0) return it;
            }
            return -1;
        };
        bool staged = false;            // this item's query rows are already in place
        for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
            const Item r = gqa_item(a, item, t == 0);
            const int64_t split0 = int64_t(r.s) * a.batch * T * a.num_q_heads;
            if (r.ntiles == 0) {
                for (int i = t; i < kRows * kD / 4; i += kSoftThreads) {
                    const int rr = i / (kD / 4), c = i % (kD / 4);
                    reinterpret_cast<float4 *>(
                        a.out_part + (split0 + row_offset(a, r, rr, Gr)) * kD)[c] =
                        make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (t < kRows) a.lse_part[split0 + row_offset(a, r, t, Gr)] = -INFINITY;
                continue;
            }
            bool w = staged || stage_q(r, ne);
            staged = false;
            // the next busy item: its query rows into L2 now, into shared
            // memory as soon as this item's last probabilities are out
            Item nx;
            const int next = next_busy(item, nx);
            if (next >= 0 && t < kRows * 4) {
                const float *qrow = a.q + row_offset(a, nx, t >> 2, Gr) * kD + (t & 3) * 32;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow));
            }
            if (t < kRows) mrow[t] = -INFINITY;
            float l_part[kRows];
#pragma unroll
            for (int h = 0; h < kRows; ++h) l_part[h] = 0.f;
            // Causal limits, from r.begin: row h (query token h / Gr) sees
            // tokens < lim0 + h / Gr, and none past the item's span.
            const int32_t span = int32_t(r.end - r.begin);
            const int64_t lim0 = r.len - (T - 1) - r.begin;
            const int64_t lim_min = lmin(lim0, span);
            const int gr_shift = __ffs(Gr) - 1;
            if (softmax_bar_or(!w)) break;

            bool ok = true;
            for (int i = 0; i < r.ntiles; ++i) {
                const uint32_t buf = tcount & 1u;
                w = pipe_wait(bar(kBarSFull + buf), (tcount >> 1) & 1u, a.status, abort_flag);
                float x[kRows];
                {
                    uint32_t hv[16], lv[16];
                    tc::fence_after_sync();
                    tc::ld16(tl + kColS + kN * buf, hv);
                    tc::ld16(tl + kColS + kN * buf + kRows, lv);
                    tc::wait_ld();
#pragma unroll
                    for (int h = 0; h < kRows; ++h)
                        x[h] = __uint_as_float(hv[h]) + __uint_as_float(lv[h]);
                }
                tc::fence_before_sync();
                mbar_arrive(bar(kBarSEmpty + buf));
                ++tcount;
                const int32_t tok = i * kM + row;           // from r.begin
                if (int64_t(i) * kM + kM > lim_min) {      // a tile some row sees in part
                    const int64_t rel = int64_t(tok) - lim0;
                    const bool in_span = tok < span;
#pragma unroll
                    for (int h = 0; h < kRows; ++h)
                        x[h] = in_span && rel < (h >> gr_shift) ? x[h] : -INFINITY;
                }
                bool need = false;
#pragma unroll
                for (int h = 0; h < kRows; ++h) need |= x[h] > mrow[h] + kSlack;
                if (softmax_bar_or(!w)) {
                    ok = false;
                    break;
                }
                if (softmax_bar_or(need)) {
#pragma unroll
                    for (int h = 0; h < kRows; ++h) {
                        float m = x[h];
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                        if (lane == h) red[quad * kRows + h] = m;
                    }
                    named_barrier_sync(1, kSoftThreads);
                    if (t < kRows) {
                        const float tm = fmaxf(fmaxf(red[t], red[kRows + t]),
                                               fmaxf(red[2 * kRows + t], red[3 * kRows + t]));
                        const float mo = mrow[t], mn = fmaxf(mo, tm);
                        aux[t] = (mo == -INFINITY || mn == -INFINITY) ? 0.f : exp2f(mo - mn);
                        mrow[t] = mn;
                    }
                    named_barrier_sync(1, kSoftThreads);
#pragma unroll
                    for (int h = 0; h < kRows; ++h) l_part[h] *= aux[h];
                    if (i > 0) {
                        // the accumulators are quiet once the previous tile's
                        // value MMAs are done
                        const bool wv = wait_pv(pcount - 1);
                        tc::fence_after_sync();
                        if (wv) {
#pragma unroll
                            for (int half = 0; half < 2; ++half) {      // hi, lo columns
                                uint32_t v[16];
                                const uint32_t ta = tl + kColO + kRows * half;
                                tc::ld16(ta, v);
                                tc::wait_ld();
#pragma unroll
                                for (int k = 0; k < 16; ++k)
                                    v[k] = __float_as_uint(__uint_as_float(v[k]) * aux[k]);
                                tc::st16(ta, v);
                            }
                            tc::wait_st();
                        }
                    }
                }
                float p[kRows];
#pragma unroll
                for (int h = 0; h < kRows; ++h) {
                    p[h] = x[h] == -INFINITY ? 0.f : ex2_approx(x[h] - mrow[h]);
                    l_part[h] += p[h];
                }
                // this P buffer was last read by the value MMAs of tile pcount-2
                if (pcount >= 2) wait_pv(pcount - 2);
                // P^T as the value MMA's K-major B operand: rows 0-15 hi,
                // 16-31 lo; this thread's token is column `row`
                {
                    uint8_t *pa = ps + (pcount & 1u) * kPBytes + (row >> 6) * (kN * 128);
                    const int c = row & 63;
#pragma unroll
                    for (int h = 0; h < kRows; ++h) {
                        const uint32_t hb = f32_to_bf16_bits(p[h]);
                        const uint32_t lb = f32_to_bf16_bits(p[h] - __uint_as_float(hb << 16));
                        *reinterpret_cast<uint16_t *>(pa + swz(h, c)) = uint16_t(hb);
                        *reinterpret_cast<uint16_t *>(pa + swz(kRows + h, c)) = uint16_t(lb);
                    }
                }
                fence_proxy_async_smem();
                tc::fence_before_sync();
                mbar_arrive(bar(kBarPFull + (pcount & 1u)));
                ++pcount;
            }
            if (!ok) break;
            // the next item's score MMAs may start while this one finishes
            if (next >= 0) {
                staged = true;
                if (softmax_bar_or(!stage_q(nx, ne + 1))) break;
            }

            // ---- epilogue: the item's last value MMAs are done
            w = wait_pv(pcount - 1);
            tc::fence_after_sync();
#pragma unroll
            for (int h = 0; h < kRows; ++h) {
                float s = l_part[h];
                s += __shfl_xor_sync(0xffffffffu, s, 16);
                s += __shfl_xor_sync(0xffffffffu, s, 8);
                s += __shfl_xor_sync(0xffffffffu, s, 4);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                if (lane == h) red[quad * kRows + h] = s;
            }
            named_barrier_sync(1, kSoftThreads);
            if (t < kRows) {
                const float l = (red[t] + red[kRows + t]) + (red[2 * kRows + t] + red[3 * kRows + t]);
                aux[t] = l > 0.f ? 1.f / l : 0.f;
                a.lse_part[split0 + row_offset(a, r, t, Gr)] =
                    l > 0.f ? (mrow[t] + log2f(l)) * kLn2 : -INFINITY;
            }
            named_barrier_sync(1, kSoftThreads);
            if (w) {
                uint32_t hv[16], lv[16];
                tc::ld16(tl + kColO, hv);
                tc::ld16(tl + kColO + kRows, lv);
                tc::wait_ld();
#pragma unroll
                for (int h = 0; h < kRows; ++h)
                    a.out_part[(split0 + row_offset(a, r, h, Gr)) * kD + row] =
                        (__uint_as_float(hv[h]) + __uint_as_float(lv[h])) * aux[h];
            }
            tc::fence_before_sync();
            mbar_arrive(bar(kBarOEmpty));
            ++ne;
            if (softmax_bar_or(!w)) break;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 gqa_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The pool as rows of 128 bf16 (`stride` elements apart), viewed 4-D as
// (64 columns, 8 rows, 2 halves at a 128-byte stride, 8-row groups); one box
// = `box` / 8 row groups of whole rows, landing as [group][half][8 rows]
// [128 B] with the 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *pool, int64_t rows, int stride, int box) {
    auto fn = gqa_encode_fn();
    if (!fn) return false;
    const cuuint64_t row_bytes = cuuint64_t(stride) * 2;
    cuuint64_t gdim[4] = {64, 8, 2, cuuint64_t(rows / 8)};
    cuuint64_t gstride[3] = {row_bytes, 128, 8 * row_bytes};
    cuuint32_t bdim[4] = {64, 8, 2, cuuint32_t(box / 8)};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool), gdim, gstride,
              bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gqa_tc_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads, int32_t q_tokens) {
    if (c.num_kv_heads <= 0 || num_q_heads % c.num_kv_heads != 0 || q_tokens < 1 ||
        kRows % q_tokens != 0)
        return false;
    // 16 rows per item, or 32 as two head groups (larger groups go to the
    // large-group kernels, which read a tile once per 64 heads)
    const int rows_per_item = num_q_heads / c.num_kv_heads * q_tokens;
    const bool pow2_bs = c.block_size >= 16 && c.block_size <= 256 &&
                         (c.block_size & (c.block_size - 1)) == 0;
    const int64_t rows = int64_t(c.num_blocks) * c.num_kv_heads * c.block_size;
    return (rows_per_item == kRows || rows_per_item == 2 * kRows) && c.head_dim_k == kD &&
           c.head_dim_v == kD && pow2_bs && rows < (int64_t(1) << 31) - 1;
}

int gqa_tc_head_groups(const pkv_cache_desc &c, int32_t num_q_heads, int32_t q_tokens) {
    return num_q_heads / c.num_kv_heads * q_tokens / kRows;
}

int gqa_tc_resident_ctas() { return sm_count() * kCtas; }

int launch_decode_gqa_tc(const DecodeArgs &a) {
    const int64_t rows = int64_t(a.cache.num_blocks) * a.cache.num_kv_heads * a.cache.block_size;
    const int box = std::min(a.cache.block_size, 64);
    CUtensorMap tk, tv;
    if (!make_map(&tk, a.k_pool, rows, kD, box) || !make_map(&tv, a.v_pool, rows, a.v_stride, box))
        return PKV_ERR_CUDA;
    static thread_local int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(decode_gqa_tc_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kSmemBytes)) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_dev = dev;
    }
    // kCtas CTAs per SM by construction (shared memory, registers and 128
    // TMEM columns each are sized for it); the persistent loop is correct
    // for any grid, so this sizes it rather than asking the occupancy
    // calculator.
    const int64_t items = int64_t(a.batch) * a.cache.num_kv_heads * a.num_splits *
                          gqa_tc_head_groups(a.cache, a.num_q_heads, a.q_tokens);
    const int grid = int(std::min<int64_t>(items, int64_t(sm_count()) * kCtas));
    if (grid <= 0) return PKV_OK;
    return launch_pdl(decode_gqa_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, a.stream, tk,
                      tv, a);
}

}  // namespace pkv
