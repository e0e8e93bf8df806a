// decode_mla_tc.cu -- paged decode attention for large query groups on the
// 5th-generation tensor cores of sm_103a (tcgen05 MMAs, fp32 accumulators
// in tensor memory).  Shape: G >= 64 query heads per KV head, e.g. the
// MLA-shaped 128 heads over one 576-dim K / 512-dim V latent head.
//
// Work item = (sequence b, KV head g, group of 64 query heads, split chunk
// s), ordered split-major so that items over the same tokens run together
// and K/V tiles shared by head groups and by sequences with a common prefix
// come from L2.  One CTA per SM walks its items tile by tile, 128 tokens a
// tile:
//   S^T[128 tok x (64 | 64)] = K_tile . [Q_hi; Q_lo]^T  (tcgen05, M=128, N=128)
//   online softmax over the 128 token lanes of S_hi + S_lo  (CUDA cores)
//   O^T[Dv x 64 heads]       += V_tile^T . P              (tcgen05, M=128, N=64)
// Tokens are the MMA's M, so the query group is N and 64 heads fit in one
// CTA's shared memory even with the fp32 query kept exact as bf16 hi + lo
// (Dk = 576: 147 KB), the two parts side by side as one N = 128 operand
// (one score MMA per k-step).  S^T (two buffers of 128 columns) and O^T
// (Dv/128 blocks of 64 columns) fill TMEM's 512 columns at Dv = 512.
//
// Warp roles (192 threads; 256 over an FP8 cache):
//   warp 0   TMA producer: K chunks [128 tok x 64 dims] (two 64-row boxes)
//            and V chunks [64 tok x 128 dims] (one box, two 64-column
//            segments), 16 KB each, through a ring of 16 KB stages (FP8:
//            the same chunks as 8 KB of codes, landed in the upper half of
//            the stage).
//   warp 1   owns the TMEM allocation; lane 0 issues every MMA and commits
//            completions to mbarriers.  It zeroes V rows past the end of a
//            sequence before they meet the tensor core (bf16).
//   warps 2-5  softmax and epilogue, one thread per TMEM lane (token row of
//            S^T, value row of O^T).  They pre-scale and split the query,
//            turn scores into probabilities (bf16 hi + lo, written in the
//            MMA's operand layout), keep per-thread partial sums, and write
//            the normalised output and LSE.
//   warps 6-7  FP8 only: converters, expanding each stage's codes in place
//            into fp16 in the bf16 chunks' layout (value rows past the end
//            written as zeros).  A stage is rewritten only after its codes
//            landed, i.e. a whole copy after its previous MMAs released it.
// The running max of each head is raised only when a score exceeds it by
// more than 8 (log2 units); then the tile max is formed across the token
// lanes and the accumulators are rescaled in TMEM.  Otherwise
// probabilities up to 2^8 are accumulated as they are -- exact in real
// arithmetic for any choice of the running max.
//
// Every wait is bounded (PKV_DEV_TIMEOUT) and all roles leave their loops
// together on an abort; out-of-range blocks and lengths are flagged in the
// status word, never dereferenced.
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

constexpr int kN = 64;                  // query heads per work item (MMA N)
constexpr int kM = 128;                 // tokens per tile (MMA M of the score product)
constexpr int kHalf = 64;               // tokens per TMA box
constexpr int kChunk = 16384;           // bytes per ring stage
constexpr int kMaxRing = 8;
constexpr int kThreads = 192;
constexpr int kSoftWarp0 = 2;           // warps 2..5: softmax and epilogue
constexpr int kSoftThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;           // S^T buffers at columns 0 and 128 (hi | lo parts)
constexpr uint32_t kColO = 256;         // O^T blocks at columns 256 + 64 j
constexpr float kSlack = 8.f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kSmemLimit = 232448;
constexpr uint32_t kIdS = tc::idesc_bf16_f32(128, 128, 0, 0);  // K-major K, K-major [Q_hi; Q_lo]
constexpr uint32_t kIdO = tc::idesc_bf16_f32(128, 64, 1, 1);   // MN-major V, MN-major P
// FP8 (E4M3) cache: the codes are turned into fp16 (exactly) by two
// converter warps, so the products run on fp16 operands.
constexpr uint32_t kIdS16 = tc::idesc_f16_f32(128, 128, 0, 0);
constexpr uint32_t kIdO16 = tc::idesc_f16_f32(128, 64, 1, 1);
constexpr int kThreadsF8 = 256;         // warps 6-7: converters
constexpr int kConvWarp0 = 6;
constexpr int kConvThreads = 64;
constexpr int kCodeBytes = 8192;        // one chunk's E4M3 codes, in the upper half of its stage

// mbarrier slots
constexpr int kBarFull = 0;             // + stage: chunk landed (TMA bytes)
constexpr int kBarEmpty = 8;            // + stage: chunk consumed (MMA commit)
constexpr int kBarSFull = 16;           // + buffer: scores ready (MMA commit)
constexpr int kBarSEmpty = 18;          // + buffer: scores read (128 arrivals)
constexpr int kBarPFull = 20;           // probabilities written (128 arrivals)
constexpr int kBarPvDone = 21;          // value MMAs of a tile done (MMA commit)
constexpr int kBarQFull = 22;           // query written (128 arrivals)
constexpr int kBarQEmpty = 23;          // score MMAs of an item done (MMA commit)
constexpr int kBarOEmpty = 24;          // accumulators read out (128 arrivals)
constexpr int kBarDrain = 25;
constexpr int kBarLanded = 26;          // + stage, FP8: the chunk's codes landed (TMA bytes)
constexpr int kNumBars = kBarLanded + kMaxRing;

struct TcShape {
    int dk_segs;      // Dk / 64
    int dv_blocks;    // Dv / 128
    int ring;         // ring stages
};

// Shared-memory map, offsets from a 1024-byte-aligned base.
struct SmemMap {
    uint32_t q_hi, q_lo, p_hi, p_lo, ring, bars, mrow, aux, red, slot, flag, end;
};
__host__ __device__ inline SmemMap smem_map(const TcShape &s) {
    SmemMap m;
    // per 64-dim segment one [128][64] K-major block: rows 0-63 the query's
    // high parts, rows 64-127 its low parts (one N = 128 operand)
    m.q_hi = 0;
    m.q_lo = 8192;
    m.p_hi = uint32_t(s.dk_segs) * 16384;
    m.p_lo = m.p_hi + kM * 128;
    m.ring = m.p_lo + kM * 128;
    m.bars = m.ring + uint32_t(s.ring) * kChunk;
    m.mrow = m.bars + kNumBars * 8;
    m.aux = m.mrow + kN * 4;
    m.red = m.aux + kN * 4;
    m.slot = m.red + 4 * kN * 4;
    m.flag = m.slot + 4;
    m.end = m.flag + 4;
    return m;
}
inline size_t tc_smem_bytes(const TcShape &s) { return 1024 + size_t(smem_map(s).end); }

__device__ __forceinline__ int64_t lmin(int64_t x, int64_t y) { return x < y ? x : y; }

// This thread's scores for heads 16c .. 16c + 15 of a tile: the product with
// the query's high parts (S^T columns 0-63) plus its low parts (64-127),
// times `mul` (1 for a bf16 cache; the item's power-of-two query scale over
// an FP8 one).
__device__ __forceinline__ void ld_scores(uint32_t ts, int c, uint32_t (&v)[16], float mul) {
    uint32_t lo[16];
    tc::ld16(ts + 16 * c, v);
    tc::ld16(ts + kN + 16 * c, lo);
    tc::wait_ld();
#pragma unroll
    for (int k = 0; k < 16; ++k)
        v[k] = __float_as_uint((__uint_as_float(v[k]) + __uint_as_float(lo[k])) * mul);
}

// One decode problem of a launch: its queries, tables, lengths, split count
// and partial outputs.  A launch runs one problem, or two in one item space
// (the cascade: every sequence's query rows over a shared prefix, and each
// sequence's rows over its own remaining tokens).
struct Problem {
    const float *q;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float *out_part, *lse_part;
    int32_t batch, num_q_heads, max_blocks, num_splits;
};

Problem problem_of(const DecodeArgs &a) {
    return Problem{a.q, a.block_tables, a.seq_lens, a.out_part, a.lse_part,
                   a.batch, a.num_q_heads, a.max_blocks, a.num_splits};
}

// Work items of a problem: (sequence, KV head, 64-head group, split).
__host__ __device__ inline int problem_items(const Problem &p, int hkv) {
    return p.batch * hkv * (p.num_q_heads / hkv / kN) * p.num_splits;
}

// The problem an item of the launch belongs to (field by field, so the
// selection stays in registers).
__device__ __forceinline__ Problem pick(const Problem &p0, const Problem &p1, bool second) {
    Problem r;
    r.q = second ? p1.q : p0.q;
    r.block_tables = second ? p1.block_tables : p0.block_tables;
    r.seq_lens = second ? p1.seq_lens : p0.seq_lens;
    r.out_part = second ? p1.out_part : p0.out_part;
    r.lse_part = second ? p1.lse_part : p0.lse_part;
    r.batch = second ? p1.batch : p0.batch;
    r.num_q_heads = second ? p1.num_q_heads : p0.num_q_heads;
    r.max_blocks = second ? p1.max_blocks : p0.max_blocks;
    r.num_splits = second ? p1.num_splits : p0.num_splits;
    return r;
}

struct TcItem {
    Problem p;
    int G;              // query heads per KV head of the item's problem
    int b, g, hg, s;
    int64_t begin, end;
    int ntiles;
};

// Item `item` of the launch: the first problem's items come first.
__device__ __forceinline__ TcItem tc_item(const DecodeArgs &a, const Problem &p0,
                                          const Problem &p1, int item, bool report) {
    TcItem r;
    const int hkv = a.cache.num_kv_heads;
    const int n0 = problem_items(p0, hkv);
    const bool second = item >= n0;
    r.p = pick(p0, p1, second);
    if (second) item -= n0;
    r.G = r.p.num_q_heads / hkv;
    const int groups = r.G / kN;
    const int per_split = r.p.batch * hkv * groups;
    r.s = item / per_split;
    int t = item % per_split;
    r.hg = t % groups;
    t /= groups;
    r.g = t % hkv;
    r.b = t / hkv;
    int64_t L = r.p.seq_lens[r.b];
    if (L < 0 || L > int64_t(r.p.max_blocks) * a.cache.block_size) {
        if (report && r.s == 0 && r.hg == 0 && r.g == 0) raise_status(a.status, PKV_DEV_SEQ_LEN);
        L = 0;
    }
    const int64_t chunk = 64 * ((L + 64LL * r.p.num_splits - 1) / (64LL * r.p.num_splits));
    r.begin = int64_t(r.s) * chunk;
    r.end = lmin(L, r.begin + chunk);
    r.ntiles = r.end > r.begin ? int((r.end - r.begin + kM - 1) / kM) : 0;
    return r;
}

// Offset of bf16 element (row, col < 64) in a [rows][64] 128-byte-swizzled
// array whose 8-row atoms are 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(int row, int col) {
    return uint32_t(row) * 128 + (uint32_t(((col >> 3) ^ row) & 7) << 4) + uint32_t(col & 7) * 2;
}

// F8: the pools hold E4M3 codes (a.k_scale, a.v_scale per KV head).  The
// producer lands each chunk's 8 KB of codes in the upper half of its ring
// stage and the converter warps expand them, exactly, into fp16 over the
// whole stage in the layout the bf16 copies have; the query and the
// probabilities are fp16 hi + lo, the query scaled by a power of two per
// item so that both parts stay inside fp16's range.
template <bool F8>
__global__ void __launch_bounds__(F8 ? kThreadsF8 : kThreads, 1)
decode_mla_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a,
                     const Problem p0, const Problem p1, const TcShape shp) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemMap sm = smem_map(shp);
    const uint32_t sb = smem_addr(base);
    float *mrow = reinterpret_cast<float *>(base + sm.mrow);   // running max per head (log2)
    float *aux = reinterpret_cast<float *>(base + sm.aux);     // rescale factor / 1 / l
    float *red = reinterpret_cast<float *>(base + sm.red);     // [4 warps][64 heads]
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(base + sm.slot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + sm.flag);
    auto bar = [&](int i) { return sb + sm.bars + 8u * uint32_t(i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bs = a.cache.block_size, hkv = a.cache.num_kv_heads;
    const int num_items = problem_items(p0, hkv) + problem_items(p1, hkv);
    const int Dk = shp.dk_segs * 64, Dv = shp.dv_blocks * 128;
    const uint64_t wlim = a.wait_ns ? a.wait_ns : kWaitLimitNs;

    if (threadIdx.x == 0) {
        for (int r = 0; r < shp.ring; ++r) {
            // bf16: the producer's arrival + TMA bytes; FP8: the converters
            mbar_init(bar(kBarFull + r), F8 ? kConvThreads : 1);
            mbar_init(bar(kBarEmpty + r), 1);
            if (F8) mbar_init(bar(kBarLanded + r), 1);
        }
        mbar_init(bar(kBarSFull), 1);
        mbar_init(bar(kBarSFull + 1), 1);
        mbar_init(bar(kBarSEmpty), kSoftThreads);
        mbar_init(bar(kBarSEmpty + 1), kSoftThreads);
        mbar_init(bar(kBarPFull), kSoftThreads);
        mbar_init(bar(kBarPvDone), 1);
        mbar_init(bar(kBarQFull), kSoftThreads);
        mbar_init(bar(kBarQEmpty), 1);
        mbar_init(bar(kBarOEmpty), kSoftThreads);
        mbar_init(bar(kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::alloc(sb + sm.slot, kTmemCols);
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
        bool ok = a.withhold == 0;              // test control: issue no copy at all
        // bf16: the chunk fills its stage; FP8: its codes fill the upper half
        // and the converters complete the stage.
        const int bar_full = F8 ? kBarLanded : kBarFull;
        // Wait for a free stage and arm it for one chunk; false on abort.
        auto acquire = [&](uint32_t &dst) -> bool {
            const bool w =
                pipe_wait(bar(kBarEmpty + stage), phase ^ 1u, a.status, abort_flag, wlim);
            if (!__all_sync(0xffffffffu, w)) return false;
            if (lane == 0)
                mbar_arrive_expect_tx(bar(bar_full + stage), F8 ? kCodeBytes : kChunk);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            dst = sb + sm.ring + uint32_t(stage) * kChunk + (F8 ? kCodeBytes : 0);
            return true;
        };
        auto advance = [&]() {
            if (++stage == shp.ring) {
                stage = 0;
                phase ^= 1u;
            }
        };
        for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
            const TcItem r = tc_item(a, p0, p1, item, false);
            if (r.ntiles == 0) continue;
            const int32_t *table = r.p.block_tables + int64_t(r.b) * r.p.max_blocks;
            // Rows of block 0 of this KV head stand in for a half tile past
            // the end (its values are masked and its V rows zeroed).
            const int32_t standin = r.g * bs;
            int32_t yp0 = standin, yp1 = standin;
            // Lane j holds the pool row of half tile (64 tokens) wbase + j:
            // one coalesced load of table entries serves 16 tiles, so the
            // ring is not left to drain behind a dependent load every tile.
            int32_t wrow = standin;
            int wbase = -64;
            for (int i = 0; i <= r.ntiles && ok; ++i) {
                int32_t y0 = standin, y1 = standin;
                if (i < r.ntiles) {
                    const int u0 = 2 * i;
                    if (u0 >= wbase + 32) {
                        wbase = u0;
                        wrow = standin;
                        const int64_t t = r.begin + int64_t(wbase + lane) * kHalf;
                        if (t < r.end) {
                            const int32_t phys = table[t / bs];
                            if (phys >= 0 && phys < a.cache.num_blocks)
                                wrow = (phys * hkv + r.g) * bs + int32_t(t % bs);
                            else
                                raise_status(a.status, PKV_DEV_BLOCK_ID);
                        }
                    }
                    y0 = __shfl_sync(0xffffffffu, wrow, u0 - wbase);
                    y1 = __shfl_sync(0xffffffffu, wrow, u0 + 1 - wbase);
                    for (int seg = 0; seg < shp.dk_segs; ++seg) {
                        uint32_t dst;
                        if (!acquire(dst)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            if constexpr (F8) {
                                // [128 rows][64 codes]: the segment's bytes of each row
                                tma_load_2d(dst, &tmap_k, seg * 64, y0, bar(bar_full + stage));
                                tma_load_2d(dst + 4096, &tmap_k, seg * 64, y1,
                                            bar(bar_full + stage));
                            } else {
                                tma_load_3d(dst, &tmap_k, 0, y0, seg, bar(kBarFull + stage));
                                tma_load_3d(dst + 8192, &tmap_k, 0, y1, seg,
                                            bar(kBarFull + stage));
                            }
                        }
                        advance();
                    }
                }
                if (i > 0 && ok) {
                    for (int vb = 0; vb < shp.dv_blocks && ok; ++vb)
                        for (int h = 0; h < 2; ++h) {
                            uint32_t dst;
                            if (!acquire(dst)) {
                                ok = false;
                                break;
                            }
                            if (lane == 0) {
                                if constexpr (F8)   // [64 rows][128 codes]
                                    tma_load_2d(dst, &tmap_v, vb * 128, h ? yp1 : yp0,
                                                bar(bar_full + stage));
                                else
                                    tma_load_3d(dst, &tmap_v, 0, h ? yp1 : yp0, 2 * vb,
                                                bar(kBarFull + stage));
                            }
                            advance();
                        }
                }
                yp0 = y0;
                yp1 = y1;
            }
        }
        // Leave no copy in flight into this CTA's shared memory.
        if (lane == 0)
            for (int s = 0; s < shp.ring; ++s)
                if (armed & (1u << s))
                    mbar_wait(bar(bar_full + s), (armed_parity >> s) & 1u, a.status);
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        int stage = 0;
        uint32_t phase = 0, tcount = 0, pcount = 0, ne = 0;
        bool ok = true;
        const uint32_t qh = sb + sm.q_hi;
        const uint32_t ph = sb + sm.p_hi, pl = sb + sm.p_lo;
        auto wait_all = [&](uint32_t b, uint32_t parity) {
            return __all_sync(0xffffffffu, pipe_wait(b, parity, a.status, abort_flag, wlim));
        };
        auto advance = [&]() {
            if (++stage == shp.ring) {
                stage = 0;
                phase ^= 1u;
            }
        };
        for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
            const TcItem r = tc_item(a, p0, p1, item, false);
            if (r.ntiles == 0) continue;
            if (!(ok = wait_all(bar(kBarQFull), ne & 1u))) break;
            for (int i = 0; i <= r.ntiles && ok; ++i) {
                if (i < r.ntiles) {
                    // ---- S^T[buf] = K_tile . [Q_hi; Q_lo]^T (sum of the halves: the scores)
                    const uint32_t buf = tcount & 1u;
                    if (!(ok = wait_all(bar(kBarSEmpty + buf), ((tcount >> 1) & 1u) ^ 1u))) break;
                    const uint32_t d = tmem + kColS + 128 * buf;
                    for (int seg = 0; seg < shp.dk_segs; ++seg) {
                        if (!(ok = wait_all(bar(kBarFull + stage), phase))) break;
                        tc::fence_after_sync();
                        if (lane == 0) {
                            const uint32_t kb = sb + sm.ring + uint32_t(stage) * kChunk;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc::mma_bf16(d, tc::smem_desc(kb + 32 * kk, 16, 1024),
                                             tc::smem_desc(qh + uint32_t(seg) * 16384 + 32 * kk,
                                                           16, 1024),
                                             F8 ? kIdS16 : kIdS, (seg | kk) != 0);
                            tc::commit(bar(kBarEmpty + stage));
                        }
                        __syncwarp();
                        advance();
                    }
                    if (!ok) break;
                    if (lane == 0) {
                        tc::commit(bar(kBarSFull + buf));
                        if (i == r.ntiles - 1) tc::commit(bar(kBarQEmpty));
                    }
                    __syncwarp();
                    ++tcount;
                }
                if (i > 0) {
                    // ---- O^T += V_tile^T . (P_hi + P_lo) for tile j
                    const int j = i - 1;
                    if (!(ok = wait_all(bar(kBarPFull), pcount & 1u))) break;
                    if (j == 0 && !(ok = wait_all(bar(kBarOEmpty), (ne & 1u) ^ 1u))) break;
                    const int64_t tok0 = r.begin + int64_t(j) * kM;
                    const int nvalid = int(lmin(kM, r.end - tok0));
                    for (int vb = 0; vb < shp.dv_blocks && ok; ++vb) {
                        const uint32_t d = tmem + kColO + 64 * uint32_t(vb);
                        for (int h = 0; h < 2; ++h) {
                            if (!(ok = wait_all(bar(kBarFull + stage), phase))) break;
                            const int first_bad = nvalid - h * kHalf;
                            if (!F8 && first_bad < kHalf) {
                                // Value rows past the end may hold any bits
                                // (NaN times a zero probability is NaN).
                                uint8_t *vt = base + sm.ring + size_t(stage) * kChunk;
                                const int r0 = first_bad > 0 ? first_bad : 0;
                                for (int idx = lane; idx < (kHalf - r0) * 16; idx += 32) {
                                    const int row = r0 + (idx >> 4), c = idx & 15;
                                    *reinterpret_cast<uint4 *>(vt + (c >> 3) * 8192 + row * 128 +
                                                               (c & 7) * 16) =
                                        make_uint4(0, 0, 0, 0);
                                }
                                fence_proxy_async_smem();
                                __syncwarp();
                            }
                            tc::fence_after_sync();
                            if (lane == 0) {
                                const uint32_t vbase = sb + sm.ring + uint32_t(stage) * kChunk;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t ad =
                                        tc::smem_desc(vbase + 2048 * kk, 8192, 1024);
                                    const uint32_t po = uint32_t(h * kHalf + 16 * kk) * 128;
                                    tc::mma_bf16(d, ad, tc::smem_desc(ph + po, 8192, 1024),
                                                 F8 ? kIdO16 : kIdO, (j | h | kk) != 0);
                                    tc::mma_bf16(d, ad, tc::smem_desc(pl + po, 8192, 1024),
                                                 F8 ? kIdO16 : kIdO, 1);
                                }
                                tc::commit(bar(kBarEmpty + stage));
                            }
                            __syncwarp();
                            advance();
                        }
                    }
                    if (!ok) break;
                    if (lane == 0) tc::commit(bar(kBarPvDone));
                    __syncwarp();
                    ++pcount;
                }
            }
            ++ne;
        }
        // Every issued MMA completes before the accumulators are released.
        if (lane == 0) {
            tc::commit(bar(kBarDrain));
            mbar_wait(bar(kBarDrain), 0, a.status);
        }
        __syncwarp();
    } else if (warp < kSoftWarp0 + 4) {
        // -------------------------------------------- softmax and epilogue
        const int t = threadIdx.x - kSoftWarp0 * 32;     // 0..127
        const int quad = warp & 3;                       // TMEM lane quadrant
        const int row = quad * 32 + lane;                // token row / value row
        const uint32_t tl = tmem + (uint32_t(quad * 32) << 16);
        const float qscale = a.scale * kLog2e;
        uint8_t *q_hi = base + sm.q_hi, *q_lo = base + sm.q_lo;
        uint8_t *p_hi = base + sm.p_hi, *p_lo = base + sm.p_lo;
        uint32_t tcount = 0, pcount = 0, ne = 0;
        // An item this CTA gives up on (a wait ran out) reports every one of
        // its rows as NaN, output and LSE; so does every later item of the CTA.
        bool abandoned = false;
        auto abandon_rows = [&](const Problem &p, int64_t orow0) {
            float4 *o = reinterpret_cast<float4 *>(p.out_part + orow0 * Dv);
            const float nan = __int_as_float(0x7fc00000);
            for (int i = t; i < kN * Dv / 4; i += kSoftThreads) o[i] = make_float4(nan, nan, nan, nan);
            if (t < kN) p.lse_part[orow0 + t] = nan;
        };
        for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
            const TcItem r = tc_item(a, p0, p1, item, t == 0);
            const int head0 = r.g * r.G + r.hg * kN;
            const int64_t orow0 = (int64_t(r.s) * r.p.batch + r.b) * r.p.num_q_heads + head0;
            if (abandoned) {
                abandon_rows(r.p, orow0);
                continue;
            }
            if (r.ntiles == 0) {
                float4 *o = reinterpret_cast<float4 *>(r.p.out_part + orow0 * Dv);
                for (int i = t; i < kN * Dv / 4; i += kSoftThreads)
                    o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t < kN) r.p.lse_part[orow0 + t] = -INFINITY;
                continue;
            }
            // ---- the group's queries, pre-scaled by scale*log2(e), as bf16 hi + lo
            // (FP8: also by the key scale and a power of two, as fp16 hi + lo)
            bool w = pipe_wait(bar(kBarQEmpty), (ne & 1u) ^ 1u, a.status, abort_flag, wlim);
            // 16-byte loads, eight in flight per thread before any is used
            // (the query is 147 KB at Dk = 576: one load at a time would
            // leave the item's first tile waiting on ~150 L2 round trips)
            const float4 *qsrc = reinterpret_cast<const float4 *>(
                r.p.q + (int64_t(r.b) * r.p.num_q_heads + head0) * Dk);
            const int n4 = kN * Dk / 4;
            float cq = qscale;     // factor of the stored query
            float mul = 1.f;       // factor of the scores read back
            if constexpr (F8) {
                // The stored query is q c 2^-e, c = scale log2(e) k_scale: 2^e
                // brings the item's largest |q c| into [2^13, 2^14), below
                // fp16's largest finite value, with the low parts of all but
                // the smallest elements still normal; the scores are read
                // back times 2^e (exact).
                float m = 0.f;
                if (w) {
                    for (int i0 = 0; i0 < n4; i0 += 8 * kSoftThreads) {
                        float4 x[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int i = i0 + u * kSoftThreads + t;
                            x[u] = i < n4 ? __ldg(qsrc + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            m = fmaxf(m, fmaxf(fmaxf(fabsf(x[u].x), fabsf(x[u].y)),
                                               fmaxf(fabsf(x[u].z), fabsf(x[u].w))));
                    }
                }
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                if (lane == 0) red[quad * kN] = m;
                w = !softmax_bar_or(!w);
                const float c = qscale * a.k_scale[r.g];
                const float big = fmaxf(fmaxf(red[0], red[kN]), fmaxf(red[2 * kN], red[3 * kN])) *
                                  fabsf(c);
                int e = 0;
                if (big > 0.f && big <= 3.402823466e38f)
                    e = min(max(int((__float_as_uint(big) >> 23) & 0xffu) - 127 - 13, -100), 100);
                cq = c * __uint_as_float(uint32_t(127 - e) << 23);
                mul = __uint_as_float(uint32_t(127 + e) << 23);
            }
            if (w) {
                for (int i0 = 0; i0 < n4; i0 += 8 * kSoftThreads) {
                    float4 x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = i0 + u * kSoftThreads + t;
                        x[u] = i < n4 ? __ldg(qsrc + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = i0 + u * kSoftThreads + t;
                        if (i >= n4) continue;
                        const int h = (4 * i) / Dk, d = (4 * i) % Dk;
                        const float x0 = x[u].x * cq, x1 = x[u].y * cq;
                        const float x2 = x[u].z * cq, x3 = x[u].w * cq;
                        uint32_t h01, h23, l01, l23;
                        if constexpr (F8) {
                            h01 = pack_f16x2(x0, x1);
                            h23 = pack_f16x2(x2, x3);
                            l01 = pack_f16x2(x0 - f16_lo_to_f32(h01), x1 - f16_hi_to_f32(h01));
                            l23 = pack_f16x2(x2 - f16_lo_to_f32(h23), x3 - f16_hi_to_f32(h23));
                        } else {
                            h01 = pack_bf16x2(x0, x1);
                            h23 = pack_bf16x2(x2, x3);
                            l01 = pack_bf16x2(x0 - bf16_lo_to_f32(h01), x1 - bf16_hi_to_f32(h01));
                            l23 = pack_bf16x2(x2 - bf16_lo_to_f32(h23), x3 - bf16_hi_to_f32(h23));
                        }
                        // four consecutive dims share one 16-byte swizzle chunk
                        const uint32_t off = uint32_t(d >> 6) * 16384 + swz(h, d & 63);
                        *reinterpret_cast<uint2 *>(q_hi + off) = make_uint2(h01, h23);
                        *reinterpret_cast<uint2 *>(q_lo + off) = make_uint2(l01, l23);
                    }
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(bar(kBarQFull));
            if (t < kN) mrow[t] = -INFINITY;
            float l_part[kN];
#pragma unroll
            for (int h = 0; h < kN; ++h) l_part[h] = 0.f;
            if (softmax_bar_or(!w)) {
                abandoned = true;
                abandon_rows(r.p, orow0);
                continue;
            }

            bool ok = true;
            for (int i = 0; i < r.ntiles; ++i) {
                // ---- scores of this thread's token for the 64 heads, read
                // from TMEM in 16-column slices (first pass: does any score
                // exceed its head's running max by more than the slack?)
                const uint32_t buf = tcount & 1u;
                const uint32_t ts = tl + kColS + 128 * buf;
                w = pipe_wait(bar(kBarSFull + buf), (tcount >> 1) & 1u, a.status, abort_flag,
                              wlim);
                tc::fence_after_sync();
                const bool valid = r.begin + int64_t(i) * kM + row < r.end;
                bool need = false;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[16];
                    ld_scores(ts, c, v, mul);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        need |= valid && __uint_as_float(v[k]) > mrow[16 * c + k] + kSlack;
                }
                if (softmax_bar_or(!w)) {
                    ok = false;
                    break;
                }
                bool pv_waited = false;
                if (softmax_bar_or(need)) {
                    // ---- raise the running max to this tile's max
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t v[16];
                        ld_scores(ts, c, v, mul);
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            float m = valid ? __uint_as_float(v[k]) : -INFINITY;
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                            if (lane == ((16 * c + k) & 31)) red[quad * kN + 16 * c + k] = m;
                        }
                    }
                    named_barrier_sync(1, kSoftThreads);
                    if (t < kN) {
                        const float tm = fmaxf(fmaxf(red[t], red[kN + t]),
                                               fmaxf(red[2 * kN + t], red[3 * kN + t]));
                        const float mo = mrow[t], mn = fmaxf(mo, tm);
                        aux[t] = mo == -INFINITY ? 0.f : exp2f(mo - mn);
                        mrow[t] = mn;
                    }
                    named_barrier_sync(1, kSoftThreads);
#pragma unroll
                    for (int h = 0; h < kN; ++h) l_part[h] *= aux[h];
                    if (i > 0) {
                        // the accumulators are quiet: tile i-1's value MMAs
                        // are done and tile i's wait for these probabilities
                        const bool wv =
                            pipe_wait(bar(kBarPvDone), pcount & 1u, a.status, abort_flag, wlim);
                        ++pcount;
                        pv_waited = true;
                        tc::fence_after_sync();
                        if (wv) {
                            for (int vb = 0; vb < shp.dv_blocks; ++vb) {
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    uint32_t v[16];
                                    const uint32_t ta = tl + kColO + 64 * uint32_t(vb) + 16 * c;
                                    tc::ld16(ta, v);
                                    tc::wait_ld();
#pragma unroll
                                    for (int k = 0; k < 16; ++k)
                                        v[k] = __float_as_uint(__uint_as_float(v[k]) *
                                                               aux[16 * c + k]);
                                    tc::st16(ta, v);
                                }
                            }
                            tc::wait_st();
                        }
                    }
                }
                if (i > 0 && !pv_waited) {
                    // tile i-1's value MMAs have finished reading the buffer
                    pipe_wait(bar(kBarPvDone), pcount & 1u, a.status, abort_flag, wlim);
                    ++pcount;
                }
                // ---- second pass: probabilities, split into bf16 hi + lo,
                // straight into the value MMA's operand layout (this token's row)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[16];
                    ld_scores(ts, c, v, mul);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int k = 8 * half + 2 * e, h = 16 * c + k;
                            const float2 m2 = *reinterpret_cast<const float2 *>(mrow + h);
                            const float x0 = valid ? __uint_as_float(v[k]) : -INFINITY;
                            const float x1 = valid ? __uint_as_float(v[k + 1]) : -INFINITY;
                            const float p0 = ex2_approx(x0 - m2.x), p1 = ex2_approx(x1 - m2.y);
                            l_part[h] += p0;
                            l_part[h + 1] += p1;
                            if constexpr (F8) {
                                hi[e] = pack_f16x2(p0, p1);
                                lo[e] = pack_f16x2(p0 - f16_lo_to_f32(hi[e]),
                                                   p1 - f16_hi_to_f32(hi[e]));
                            } else {
                                hi[e] = pack_bf16x2(p0, p1);
                                lo[e] = pack_bf16x2(p0 - bf16_lo_to_f32(hi[e]),
                                                    p1 - bf16_hi_to_f32(hi[e]));
                            }
                        }
                        const int chunk = 2 * c + half;
                        const uint32_t off =
                            uint32_t(row) * 128 + (uint32_t((chunk ^ row) & 7) << 4);
                        *reinterpret_cast<uint4 *>(p_hi + off) =
                            make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(p_lo + off) =
                            make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                tc::fence_before_sync();
                mbar_arrive(bar(kBarSEmpty + buf));
                ++tcount;
                fence_proxy_async_smem();
                tc::fence_before_sync();
                mbar_arrive(bar(kBarPFull));
            }
            if (!ok) {
                abandoned = true;
                abandon_rows(r.p, orow0);
                continue;
            }

            // ---- epilogue: the item's last value MMAs are complete
            w = pipe_wait(bar(kBarPvDone), pcount & 1u, a.status, abort_flag, wlim);
            ++pcount;
            tc::fence_after_sync();
#pragma unroll
            for (int h = 0; h < kN; ++h) {
                float s = l_part[h];
                s += __shfl_xor_sync(0xffffffffu, s, 16);
                s += __shfl_xor_sync(0xffffffffu, s, 8);
                s += __shfl_xor_sync(0xffffffffu, s, 4);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                if (lane == (h & 31)) red[quad * kN + h] = s;
            }
            named_barrier_sync(1, kSoftThreads);
            if (t < kN) {
                const float l = (red[t] + red[kN + t]) + (red[2 * kN + t] + red[3 * kN + t]);
                // FP8: the values' scale goes with 1 / l
                aux[t] = l > 0.f ? (F8 ? a.v_scale[r.g] : 1.f) / l : 0.f;
                r.p.lse_part[orow0 + t] = l > 0.f ? (mrow[t] + log2f(l)) * kLn2 : -INFINITY;
            }
            named_barrier_sync(1, kSoftThreads);
            if (w) {
                for (int vb = 0; vb < shp.dv_blocks; ++vb) {
                    float *orow = r.p.out_part + orow0 * Dv + vb * 128 + row;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t v[16];
                        tc::ld16(tl + kColO + 64 * uint32_t(vb) + 16 * c, v);
                        tc::wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            orow[int64_t(16 * c + k) * Dv] =
                                __uint_as_float(v[k]) * aux[16 * c + k];
                    }
                }
            }
            tc::fence_before_sync();
            mbar_arrive(bar(kBarOEmpty));
            ++ne;
            if (softmax_bar_or(!w)) {
                abandoned = true;
                abandon_rows(r.p, orow0);
            }
        }
    } else {
        if constexpr (F8) {
            // ------------------------------------------ E4M3 -> fp16 converters
            // A chunk's codes are 512 pieces of 16, eight per thread: piece p
            // of a key chunk ([128 rows][64 codes]) is row p / 4, dims
            // 16 (p % 4) .. + 15 of the segment; of a value chunk ([64 rows]
            // [128 codes]) row p / 8, dims 16 (p % 8) .. + 15 of the block.
            // Eight consecutive threads read 128 consecutive bytes and store
            // to disjoint banks (value pieces of the second 64 dims store
            // their two halves in the other order).  Value rows past the end
            // of the sequence are written as zeros (any bits may sit there,
            // and NaN times a zero probability is NaN).
            const int t = threadIdx.x - kConvWarp0 * 32;    // 0..63
            int stage = 0;
            uint32_t phase = 0;
            auto convert = [&](bool is_v, int keep) -> bool {
                const bool w =
                    pipe_wait(bar(kBarLanded + stage), phase, a.status, abort_flag, wlim);
                uint8_t *st = base + sm.ring + size_t(stage) * kChunk;
                uint4 cd[8];
                if (w) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        cd[k] = *reinterpret_cast<const uint4 *>(st + kCodeBytes +
                                                                 16 * (t + 64 * k));
                }
                // every code is read before fp16 values overwrite the stage
                if (bar_red_or(2, kConvThreads, !w)) return false;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int p = t + 64 * k;
                    int row, q2;
                    uint32_t off;
                    bool zero = false, swap = false;
                    if (is_v) {
                        row = p >> 3;
                        const int q = p & 7;
                        off = uint32_t(q >> 2) * 8192 + uint32_t(row) * 128;
                        q2 = 2 * (q & 3);
                        zero = row >= keep;
                        swap = (q & 4) != 0;
                    } else {
                        row = p >> 2;
                        off = uint32_t(row) * 128;
                        q2 = 2 * (p & 3);
                    }
                    const uint2 f0 = e4m3x4_to_f16x4(cd[k].x), f1 = e4m3x4_to_f16x4(cd[k].y);
                    const uint2 f2 = e4m3x4_to_f16x4(cd[k].z), f3 = e4m3x4_to_f16x4(cd[k].w);
                    uint4 lo = make_uint4(f0.x, f0.y, f1.x, f1.y);
                    uint4 hi = make_uint4(f2.x, f2.y, f3.x, f3.y);
                    if (zero) lo = hi = make_uint4(0, 0, 0, 0);
                    const uint32_t o0 = off + (uint32_t((q2 ^ row) & 7) << 4);
                    const uint32_t o1 = off + (uint32_t(((q2 + 1) ^ row) & 7) << 4);
                    *reinterpret_cast<uint4 *>(st + (swap ? o1 : o0)) = swap ? hi : lo;
                    *reinterpret_cast<uint4 *>(st + (swap ? o0 : o1)) = swap ? lo : hi;
                }
                fence_proxy_async_smem();
                mbar_arrive(bar(kBarFull + stage));
                if (++stage == shp.ring) {
                    stage = 0;
                    phase ^= 1u;
                }
                return true;
            };
            // the producer's order of chunks
            bool ok = true;
            for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
                const TcItem r = tc_item(a, p0, p1, item, false);
                if (r.ntiles == 0) continue;
                for (int i = 0; i <= r.ntiles && ok; ++i) {
                    if (i < r.ntiles)
                        for (int seg = 0; seg < shp.dk_segs && ok; ++seg) ok = convert(false, kM);
                    if (i > 0) {
                        const int64_t tok0 = r.begin + int64_t(i - 1) * kM;
                        const int nvalid = int(lmin(kM, r.end - tok0));
                        for (int vb = 0; vb < shp.dv_blocks && ok; ++vb)
                            for (int h = 0; h < 2 && ok; ++h)
                                ok = convert(true, nvalid - h * kHalf);
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
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

// The pool as rows of `dim` bf16 (`stride` elements apart), viewed 3-D as
// (64 columns, rows, dim/64 segments at a 128-byte stride); one box = 64
// rows x `segs` segments, landing segment-major with the 128-byte swizzle.
bool make_box_map(CUtensorMap *map, const void *pool, int64_t rows, int dim, int stride,
                  int segs) {
    auto fn = tc_encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[3] = {64, cuuint64_t(rows), cuuint64_t(dim / 64)};
    cuuint64_t gstride[2] = {cuuint64_t(stride) * 2, 128};
    cuuint32_t box[3] = {64, cuuint32_t(kHalf), cuuint32_t(segs)};
    cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), gdim, gstride,
              box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The E4M3 pool as rows of `dim` one-byte codes (`stride` bytes apart); one
// box = 64 rows x `box_x` codes, unswizzled ([64][box_x] in shared memory).
bool make_code_map(CUtensorMap *map, const void *pool, int64_t rows, int dim, int stride,
                   int box_x) {
    auto fn = tc_encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {cuuint64_t(dim), cuuint64_t(rows)};
    cuuint64_t gstride[1] = {cuuint64_t(stride)};
    cuuint32_t box[2] = {cuuint32_t(box_x), cuuint32_t(kHalf)};
    cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), gdim, gstride, box,
              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

TcShape tc_shape(const pkv_cache_desc &c) {
    TcShape s{c.head_dim_k / 64, c.head_dim_v / 128, 0};
    const size_t fixed = tc_smem_bytes(s);
    const int ring = int((kSmemLimit - std::min<size_t>(fixed, kSmemLimit)) / kChunk);
    s.ring = std::min(ring, kMaxRing);
    return s;
}

}  // namespace

bool mla_tc_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads) {
    const int G = num_q_heads / c.num_kv_heads;
    const bool pow2_bs = c.block_size >= kHalf && c.block_size <= 256 &&
                         (c.block_size & (c.block_size - 1)) == 0;
    const int64_t rows = int64_t(c.num_blocks) * c.num_kv_heads * c.block_size;
    if (G % kN != 0 || !pow2_bs || rows >= (int64_t(1) << 31) - 1) return false;
    if (c.head_dim_k % 64 != 0 || c.head_dim_k < 64 || c.head_dim_v % 128 != 0 ||
        c.head_dim_v > 512)
        return false;
    return tc_shape(c).ring >= 2;
}

bool mla_tc_e4m3_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads) {
    return mla_tc_kernel_supports(c, num_q_heads);
}

int32_t mla_tc_work_units(const pkv_cache_desc &c, int32_t batch, int32_t num_q_heads) {
    return batch * num_q_heads / kN;
}

namespace {
// One launch over the problems' items together (p1.batch = 0: one problem).
template <bool F8>
int launch_problems(const DecodeArgs &a, const Problem &p0, const Problem &p1) {
    const TcShape shp = tc_shape(a.cache);
    const int64_t rows = int64_t(a.cache.num_blocks) * a.cache.num_kv_heads * a.cache.block_size;
    CUtensorMap tk, tv;
    const bool maps =
        F8 ? make_code_map(&tk, a.k_pool, rows, a.cache.head_dim_k, a.cache.head_dim_k, 64) &&
                 make_code_map(&tv, a.v_pool, rows, a.cache.head_dim_v, a.v_stride, 128)
           : make_box_map(&tk, a.k_pool, rows, a.cache.head_dim_k, a.cache.head_dim_k, 1) &&
                 make_box_map(&tv, a.v_pool, rows, a.cache.head_dim_v, a.v_stride, 2);
    if (!maps) return PKV_ERR_CUDA;
    const size_t smem = tc_smem_bytes(shp);
    static thread_local int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(decode_mla_tc_kernel<F8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemLimit) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_dev = dev;
    }
    const int hkv = a.cache.num_kv_heads;
    const int64_t items = int64_t(problem_items(p0, hkv)) + problem_items(p1, hkv);
    const int grid = int(std::min<int64_t>(items, sm_count()));
    if (grid <= 0) return PKV_OK;
    return launch_pdl(decode_mla_tc_kernel<F8>, dim3(grid), dim3(F8 ? kThreadsF8 : kThreads),
                      smem, a.stream, tk, tv, a, p0, p1, shp);
}
}  // namespace

int launch_decode_mla_tc(const DecodeArgs &a) {
    Problem none = problem_of(a);
    none.batch = 0;
    return launch_problems<false>(a, problem_of(a), none);
}

int launch_decode_mla_tc_two(const DecodeArgs &first, const DecodeArgs &second) {
    return launch_problems<false>(first, problem_of(first), problem_of(second));
}

int launch_decode_mla_tc_e4m3(const DecodeArgs &a) {
    Problem none = problem_of(a);
    none.batch = 0;
    return launch_problems<true>(a, problem_of(a), none);
}

}  // namespace pkv
