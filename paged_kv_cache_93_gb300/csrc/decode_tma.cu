// decode_tma.cu -- paged decode attention for GQA shapes on sm_103a.
//
// Work item = (sequence b, KV head g, split s): the chunk of tokens
// [s*C, min(L, (s+1)*C)) of sequence b, C = 64 * ceil(L / (64 * S)), for all
// G query rows that share KV head g: the Hq / Hkv query heads of the group,
// times T query tokens when a step brings T new tokens per sequence (row
// (t, h) then attends causally: to the first L - T + 1 + t tokens).  A persistent grid walks the
// items round-robin; each CTA has one producer warp and W consumer warps,
// and several CTAs share an SM.
//
// Producer warp: reads block-table entries (one per lane, 32 segments at a
// time) and moves each segment -- the (block, KV head) tile, or 16*W tokens of
// it when blocks are longer -- with ONE TMA tensor copy per tensor: the tile
// is contiguous in HBM, and the copy lands it as 64-column halves, each a
// 128-byte-swizzled [rows x 128 B] array, so ldmatrix reads are bank-conflict
// free.  A stage holds 16*W tokens of K and of V.  Segments past the end of
// the chunk (and table entries outside the pool) are fetched from block 0 of
// the same KV head, a row that always exists; the consumers mask those
// tokens' scores and zero their value rows, so whatever that row holds never
// reaches the result.  Stage hand-off uses mbarriers (full: producer
// expect_tx + TMA bytes; empty: one arrival per consumer warp).  Every wait is
// bounded.
//
// Consumer warps: warp w owns tokens [16w, 16w+16) of every stage.  Scores are
// computed transposed, S^T[16 tokens x 8 cols] = K[16 x D] . [q_hi | q_lo]^T,
// with bf16 mma.sync (fp32 accumulate); the fp32 query is split into two bf16
// terms (hi + lo) packed side by side in the N dimension, so the split costs
// no extra MMA and scores keep ~16 mantissa bits of the query.  The online
// softmax runs in base 2 (query pre-scaled by scale*log2 e); probabilities
// are split the same way (p_hi | p_lo) and the value product is
// O^T[D x 8 cols] += V^T[D x 16] . [p_hi | p_lo]^T, again one MMA per 16 rows
// of D.  At the end of an item the warps' (m, l, O) are merged through shared
// memory and written as that chunk's partial (or final) result.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_math.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kRowBytes = 128;     // one 64-column half-row of bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// D: head dim (64 or 128); G: query rows per KV head (1, 2, 4, 8, 16);
// W: consumer warps per CTA; NSTAGES: pipeline depth; MINB: CTAs per SM the
// register allocation must allow.
template <int D, int G, int W, int NSTAGES, int MINB>
struct Cfg {
    static constexpr int kStageTokens = 16 * W;
    static constexpr int kThreads = (W + 1) * 32;
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = kStageTokens * D * 2;    // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kNT = (2 * G + 7) / 8;                // 8-column n-tiles (hi|lo)
    static constexpr int kSlots = G >= 8 ? G / 4 : 2;          // query rows held per lane
    static constexpr int kKSteps = D / 16;
    static constexpr int kMTiles = D / 16;
    static constexpr int kMergeFloats = W * (2 * G + G * D);
    static constexpr int kPbufFloats = W * 16 * G;
    static constexpr size_t kSmemBytes = 1024 + size_t(NSTAGES) * kStageBytes +
                                         2 * NSTAGES * sizeof(uint64_t) +
                                         sizeof(float) * (kMergeFloats + kPbufFloats) + 16;
    static_assert(NSTAGES <= 32, "stage bit masks are 32 bits wide");
    static_assert(W == 1 || W == 2 || W == 4 || W == 8, "stages must tile a 32-segment window");
};

__device__ __forceinline__ int64_t lmin(int64_t x, int64_t y) { return x < y ? x : y; }
__device__ __forceinline__ int64_t lmax(int64_t x, int64_t y) { return x > y ? x : y; }

struct ItemRange {
    int b, g, s;
    int64_t len;                 // the sequence's token count (0 if invalid)
    int64_t begin, end;
    int nstages;
};

__device__ __forceinline__ ItemRange item_range(const DecodeArgs &a, int item, int stage_tokens,
                                                bool report) {
    ItemRange r;
    r.s = item % a.num_splits;
    const int t = item / a.num_splits;
    r.g = t % a.cache.num_kv_heads;
    r.b = t / a.cache.num_kv_heads;
    int64_t L = a.seq_lens[r.b];
    if (L < 0 || L > int64_t(a.max_blocks) * a.cache.block_size) {
        if (report && r.s == 0) raise_status(a.status, PKV_DEV_SEQ_LEN);
        L = 0;
    } else if (L < a.flag_below && report && r.s == 0) {
        // fewer stored tokens than the step's new ones: the rows of the
        // missing tokens stay empty
        raise_status(a.status, PKV_DEV_SEQ_LEN);
    }
    const int64_t chunk = 64 * ((L + 64LL * a.num_splits - 1) / (64LL * a.num_splits));
    r.len = L;
    r.begin = int64_t(r.s) * chunk;
    r.end = lmin(L, r.begin + chunk);
    r.nstages = r.end > r.begin ? int((r.end - r.begin + stage_tokens - 1) / stage_tokens) : 0;
    return r;
}

// Row `row` (0..G-1) of an item -> offset of its query / output row in
// units of one head vector: query token t = row / Gr of sequence b, head
// g * Gr + row % Gr (Gr = G / T query heads per KV head).
__device__ __forceinline__ int64_t row_offset(const DecodeArgs &a, int b, int g, int row, int Gr) {
    const int t = row / Gr, h = row - t * Gr;
    return (int64_t(b) * a.q_tokens + t) * a.num_q_heads + int64_t(g) * Gr + h;
}

// Column n (0..8*NT-1) of the packed [hi | lo] operand -> (head, is_lo), or
// head = -1 for a zero padding column.
template <int G>
__device__ __forceinline__ int col_head(int n, bool &is_lo) {
    if constexpr (G >= 8) {
        is_lo = n >= G;
        return n & (G - 1);
    } else {
        is_lo = n >= G;
        return n < 2 * G ? (n % G) : -1;
    }
}

// Shared-memory layout of one stage's K (or V): segment-major, each segment
// [half][seg_rows][128 B] with the 16-byte chunk index XOR-ed with (row & 7).
// Segments and halves start on 1 KiB boundaries (seg_rows >= 8), so the
// hardware's 128-byte swizzle pattern is exactly (row & 7).
struct StageLayout {
    uint32_t seg_shift;   // log2(rows per segment)
    uint32_t seg_bytes;   // bytes of one segment (all halves)
    uint32_t half_bytes;  // bytes of one half of a segment
    __device__ __forceinline__ uint32_t row_base(int row) const {
        return (uint32_t(row) >> seg_shift) * seg_bytes +
               (uint32_t(row) & ((1u << seg_shift) - 1)) * kRowBytes;
    }
};

template <int D>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, int32_t row,
                                         uint32_t bar) {
    if constexpr (D == 128)
        tma_load_3d(dst, map, 0, row, 0, bar);
    else
        tma_load_2d(dst, map, 0, row, bar);
}

template <int D, int G, int W, int NSTAGES, int MINB>
__global__ void __launch_bounds__((W + 1) * 32, MINB)
decode_tma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
    using C = Cfg<D, G, W, NSTAGES, MINB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + size_t(NSTAGES) * C::kStageBytes);
    uint64_t *empty_bar = full_bar + NSTAGES;
    float *merge = reinterpret_cast<float *>(empty_bar + NSTAGES);
    float *pbuf = merge + C::kMergeFloats;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(pbuf + C::kPbufFloats);
    volatile int *stop_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_items = a.batch * a.cache.num_kv_heads * a.num_splits;
    const int bs = a.cache.block_size;
    const int hkv = a.cache.num_kv_heads;
    const uint64_t wlim = a.wait_ns ? a.wait_ns : kWaitLimitNs;
    const int seg_rows = bs < C::kStageTokens ? bs : C::kStageTokens;
    const uint32_t seg_shift = 31 - __clz(seg_rows);
    const StageLayout lay{seg_shift, uint32_t(seg_rows) * D * 2, uint32_t(seg_rows) * kRowBytes};

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGES; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), W);
        }
        *abort_flag = 0;
        *stop_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Everything above overlaps the previous kernel's tail; inputs are read
    // only after it has finished.
    pdl_launch_dependents();
    pdl_wait();

    if (warp == W) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        const int segs_per_stage = C::kStageTokens / seg_rows;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t armed = 0, armed_parity = 0;   // per stage: ever armed / parity armed last
        bool ok = a.withhold == 0;              // test control: issue no copy at all
        for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
            const ItemRange r = item_range(a, item, C::kStageTokens, false);
            const int total_segs = r.nstages * segs_per_stage;
            const int32_t *table = a.block_tables + int64_t(r.b) * a.max_blocks;
            for (int base = 0; base < total_segs && ok; base += 32) {
                // Lane i resolves segment base + i to a global row; block 0
                // of this KV head stands in for segments without a token.
                int32_t y = r.g * bs;
                const int sg = base + lane;
                if (sg < total_segs) {
                    const int64_t ts = r.begin + int64_t(sg) * seg_rows;
                    if (ts < r.end) {
                        const int32_t phys = table[ts / bs];
                        if (phys >= 0 && phys < a.cache.num_blocks)
                            y = (phys * hkv + r.g) * bs + int32_t(ts % bs);
                        else
                            raise_status(a.status, PKV_DEV_BLOCK_ID);
                    }
                }
                const int nseg = min(32, total_segs - base);
                for (int k = 0; k < nseg; k += segs_per_stage) {
                    const uint32_t eb = smem_addr(&empty_bar[stage]);
                    const uint32_t fb = smem_addr(&full_bar[stage]);
                    int fail = 0;
                    if (lane == 0) fail = !mbar_wait(eb, phase ^ 1u, a.status, wlim) || *abort_flag;
                    if (__shfl_sync(0xffffffffu, fail, 0)) {
                        if (lane == 0) *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(fb, C::kStageBytes);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    const uint32_t kdst = smem_addr(smem + size_t(stage) * C::kStageBytes);
                    const uint32_t vdst = kdst + C::kTileBytes;
                    for (int q = 0; q < segs_per_stage; ++q) {
                        const int32_t yq = __shfl_sync(0xffffffffu, y, k + q);
                        if (lane == 0) {
                            tma_tile<D>(kdst + q * lay.seg_bytes, &tmap_k, yq, fb);
                            tma_tile<D>(vdst + q * lay.seg_bytes, &tmap_v, yq, fb);
                        }
                    }
                    if (++stage == NSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        // Do not leave while copies issued by this CTA may still be landing
        // in its shared memory (matters only if the consumers gave up).
        if (lane == 0)
            for (int s = 0; s < NSTAGES; ++s)
                if (armed & (1u << s))
                    mbar_wait(smem_addr(&full_bar[s]), (armed_parity >> s) & 1u, a.status);
        return;
    }

    // -------------------------------------------------------------- consumers
    float *pw = pbuf + warp * 16 * G;                  // this warp's p transpose buffer
    float *mw = merge + warp * (2 * G + G * D);         // this warp's (m, l, O) for the merge
    const int r0 = lane >> 2;                           // token row (and +8) inside the slice
    const int tq = lane & 3;
    // Query-row slots of this lane: columns 2*tq and 2*tq+1 of each packed
    // hi tile (G >= 8: G/8 hi tiles, so G/4 slots; G <= 4: two slots, the
    // hi and lo columns of a row meeting through a shuffle).
    constexpr int NS = C::kSlots;
    int slot_head[NS];
    bool slot_ok[NS];
    if constexpr (G >= 8) {
#pragma unroll
        for (int j = 0; j < NS; ++j) {
            slot_head[j] = 8 * (j >> 1) + 2 * tq + (j & 1);
            slot_ok[j] = true;
        }
    } else if constexpr (G == 4) {
        slot_head[0] = 2 * (tq & 1); slot_head[1] = 2 * (tq & 1) + 1; slot_ok[0] = slot_ok[1] = true;
    } else if constexpr (G == 2) {
        slot_head[0] = 0; slot_head[1] = 1; slot_ok[0] = slot_ok[1] = tq < 2;
    } else {
        slot_head[0] = 0; slot_head[1] = 0; slot_ok[0] = tq == 0; slot_ok[1] = false;
    }
    const float qscale = a.scale * kLog2e;
    // ldmatrix row addresses inside a stage (constant per lane).
    const int krow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;   // A = K, non-transposed
    const int vrow = 16 * warp + (lane & 7) + (lane >> 4) * 8;         // A = V^T, transposed
    const uint32_t koff = lay.row_base(krow), voff = lay.row_base(vrow);
    const int ksw = krow & 7, vsw = vrow & 7;

    const int T = a.q_tokens, Gr = G / a.q_tokens;    // query tokens, heads per KV head
    // An item this CTA gives up on (a wait ran out) reports every one of its
    // rows as NaN, output and LSE; so does every later item of the CTA.
    auto abandon_rows = [&](const ItemRange &r) {
        const int64_t split0 = int64_t(r.s) * a.batch * T * a.num_q_heads;
        for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
            const int head = idx / D, d = idx % D;
            const int64_t orow = split0 + row_offset(a, r.b, r.g, head, Gr);
            a.out_part[orow * D + d] = __int_as_float(0x7fc00000);
            if (d == 0) a.lse_part[orow] = __int_as_float(0x7fc00000);
        }
    };

    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
        const ItemRange r = item_range(a, item, C::kStageTokens, warp == 0 && lane == 0);
        if (!ok) {
            abandon_rows(r);
            continue;
        }

        // Query fragments: B operand of S^T = K . Q^T, columns [q_hi | q_lo].
        uint32_t qf[C::kKSteps][C::kNT][2];
        {
#pragma unroll
            for (int nt = 0; nt < C::kNT; ++nt) {
                bool is_lo;
                const int head = col_head<G>(nt * 8 + r0, is_lo);
                const float *qrow =
                    a.q + (head >= 0 ? row_offset(a, r.b, r.g, head, Gr) : 0) * D;
#pragma unroll
                for (int ks = 0; ks < C::kKSteps; ++ks) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float v[2] = {0.f, 0.f};
                        if (head >= 0) {
                            const int d = ks * 16 + 2 * tq + half * 8;
                            const float2 x = *reinterpret_cast<const float2 *>(qrow + d);
                            const float xs[2] = {x.x * qscale, x.y * qscale};
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float hi = __uint_as_float(f32_to_bf16_bits(xs[e]) << 16);
                                v[e] = is_lo ? xs[e] - hi : hi;
                            }
                        }
                        qf[ks][nt][half] = pack_bf16x2(v[0], v[1]);
                    }
                }
            }
        }

        float acc[C::kMTiles][C::kNT][4];
#pragma unroll
        for (int mt = 0; mt < C::kMTiles; ++mt)
#pragma unroll
            for (int nt = 0; nt < C::kNT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
        float m2[NS], l2[NS];
        int64_t lim[NS];          // causal limit of the slot's row (T > 1)
#pragma unroll
        for (int j = 0; j < NS; ++j) {
            m2[j] = -INFINITY;
            l2[j] = 0.f;
            lim[j] = r.len - (T - 1 - slot_head[j] / Gr);
        }

        for (int st = 0; st < r.nstages && ok; ++st) {
            const uint32_t fb = smem_addr(&full_bar[stage]);
            const bool waited = mbar_wait(fb, phase, a.status, wlim);
            if (__any_sync(0xffffffffu, !waited || *abort_flag)) {
                if (lane == 0) *abort_flag = 1;
                ok = false;
                break;
            }
            uint8_t *kstage = smem + size_t(stage) * C::kStageBytes;
            const uint32_t kbase = smem_addr(kstage);
            const uint32_t vbase = kbase + C::kTileBytes;
            const int64_t tok0 = r.begin + int64_t(st) * C::kStageTokens + 16 * warp;
            const int nvalid = int(lmax(0, lmin(16, r.end - tok0)));
            if (nvalid < 16) {
                // Rows past the end may hold any bits (unused slots of the last
                // block, or the stand-in block): zero this warp's V rows there
                // so 0 * garbage cannot reach the accumulator.
                const int nrows = 16 - nvalid;
                for (int idx = lane; idx < nrows * C::kHalves * 8; idx += 32) {
                    const int row = 16 * warp + nvalid + idx / (C::kHalves * 8);
                    const int rest = idx % (C::kHalves * 8);
                    *reinterpret_cast<uint4 *>(kstage + C::kTileBytes + lay.row_base(row) +
                                               (rest / 8) * lay.half_bytes + (rest % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (nvalid > 0) {
                // ---- S^T = K . [q_hi | q_lo]^T  (two accumulator sets for ILP
                // when there are few n-tiles; G = 16 has four independent ones)
                constexpr int kSets = C::kNT >= 4 ? 1 : 2;
                float sacc[kSets][C::kNT][4];
#pragma unroll
                for (int x = 0; x < kSets; ++x)
#pragma unroll
                    for (int nt = 0; nt < C::kNT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sacc[x][nt][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < C::kKSteps; ++ks) {
                    const int chunk = (ks & 3) * 2 + (lane >> 4);
                    const uint32_t addr =
                        kbase + koff + (ks >> 2) * lay.half_bytes + ((chunk ^ ksw) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < C::kNT; ++nt)
                        mma_bf16_16816(sacc[ks % kSets][nt], a0, a1, a2, a3, qf[ks][nt][0],
                                       qf[ks][nt][1]);
                }
                float sraw[C::kNT][4];
#pragma unroll
                for (int nt = 0; nt < C::kNT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sraw[nt][e] = kSets == 2 ? sacc[0][nt][e] + sacc[kSets - 1][nt][e]
                                                 : sacc[0][nt][e];

                // ---- combine hi + lo: s[i][j] for token r0 + 8i, row slot j
                float s[2][NS];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
#pragma unroll
                    for (int j = 0; j < NS; ++j) {
                        float v;
                        if constexpr (G >= 8) {
                            v = sraw[j >> 1][2 * i + (j & 1)] + sraw[(j >> 1) + G / 8][2 * i + (j & 1)];
                        } else if constexpr (G == 4) {
                            v = sraw[0][2 * i + j] + __shfl_xor_sync(0xffffffffu, sraw[0][2 * i + j], 2);
                        } else if constexpr (G == 2) {
                            v = sraw[0][2 * i + j] + __shfl_xor_sync(0xffffffffu, sraw[0][2 * i + j], 1);
                        } else {
                            v = sraw[0][2 * i] + sraw[0][2 * i + 1];
                        }
                        const bool valid_tok =
                            (r0 + 8 * i) < nvalid && tok0 + r0 + 8 * i < lim[j];
                        s[i][j] = slot_ok[j] ? (valid_tok ? v : -INFINITY) : 0.f;
                    }
                }
                // ---- online softmax (base 2).  A row may have no token yet
                // (causal rows of a multi-token step): its max stays -inf
                // and it takes nothing from this slice.
                float alpha[NS], p[2][NS];
#pragma unroll
                for (int j = 0; j < NS; ++j) {
                    float mx = fmaxf(s[0][j], s[1][j]);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float m_new = fmaxf(m2[j], mx);
                    const float m_use = m_new == -INFINITY ? 0.f : m_new;
                    alpha[j] = ex2_approx(m2[j] - m_use);
                    p[0][j] = ex2_approx(s[0][j] - m_use);
                    p[1][j] = ex2_approx(s[1][j] - m_use);
                    l2[j] = l2[j] * alpha[j] + p[0][j] + p[1][j];
                    m2[j] = m_new;
                }
#pragma unroll
                for (int mt = 0; mt < C::kMTiles; ++mt)
#pragma unroll
                    for (int nt = 0; nt < C::kNT; ++nt) {
                        float a0, a1;
                        if constexpr (G >= 8) {
                            a0 = alpha[2 * (nt % (G / 8))];
                            a1 = alpha[2 * (nt % (G / 8)) + 1];
                        } else {
                            a0 = alpha[0];
                            a1 = (G == 1) ? alpha[0] : alpha[1];
                        }
                        acc[mt][nt][0] *= a0; acc[mt][nt][1] *= a1;
                        acc[mt][nt][2] *= a0; acc[mt][nt][3] *= a1;
                    }

                // ---- P^T fragments through the per-warp transpose buffer
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < NS; ++j)
                        if (slot_ok[j]) pw[(r0 + 8 * i) * G + slot_head[j]] = p[i][j];
                __syncwarp();
                uint32_t pf[C::kNT][2];
#pragma unroll
                for (int nt = 0; nt < C::kNT; ++nt) {
                    bool is_lo;
                    const int head = col_head<G>(nt * 8 + r0, is_lo);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float v[2] = {0.f, 0.f};
                        if (head >= 0) {
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float x = pw[(2 * tq + e + 8 * half) * G + head];
                                const float hi = __uint_as_float(f32_to_bf16_bits(x) << 16);
                                v[e] = is_lo ? x - hi : hi;
                            }
                        }
                        pf[nt][half] = pack_bf16x2(v[0], v[1]);
                    }
                }

                // ---- O^T += V^T . [p_hi | p_lo]^T
#pragma unroll
                for (int mt = 0; mt < C::kMTiles; ++mt) {
                    const int chunk = (mt & 3) * 2 + ((lane >> 3) & 1);
                    const uint32_t addr =
                        vbase + voff + (mt >> 2) * lay.half_bytes + ((chunk ^ vsw) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_trans(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < C::kNT; ++nt)
                        mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, pf[nt][0], pf[nt][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
            if (++stage == NSTAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }

        // ---- per-warp finalize: full l, hi+lo columns combined
#pragma unroll
        for (int j = 0; j < NS; ++j) {
            l2[j] += __shfl_xor_sync(0xffffffffu, l2[j], 4);
            l2[j] += __shfl_xor_sync(0xffffffffu, l2[j], 8);
            l2[j] += __shfl_xor_sync(0xffffffffu, l2[j], 16);
        }
#pragma unroll
        for (int mt = 0; mt < C::kMTiles; ++mt) {
            if constexpr (G >= 8) {
                // hi tile nh and its lo tile nh + G/8: rows 8*nh + 2*tq + c
#pragma unroll
                for (int nh = 0; nh < G / 8; ++nh)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 2 * nh + (e & 1);
                        mw[2 * G + slot_head[j] * D + mt * 16 + r0 + 8 * (e >> 1)] =
                            acc[mt][nh][e] + acc[mt][nh + G / 8][e];
                    }
            } else {
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (G == 4) {
                        o[e] = acc[mt][0][e] + __shfl_xor_sync(0xffffffffu, acc[mt][0][e], 2);
                    } else if constexpr (G == 2) {
                        o[e] = acc[mt][0][e] + __shfl_xor_sync(0xffffffffu, acc[mt][0][e], 1);
                    } else {
                        o[e] = acc[mt][0][e & 2] + acc[mt][0][(e & 2) + 1];
                    }
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        if (slot_ok[j])
                            mw[2 * G + slot_head[j] * D + mt * 16 + r0 + 8 * i] = o[2 * i + j];
            }
        }
        if (lane < 4) {
#pragma unroll
            for (int j = 0; j < NS; ++j)
                if (slot_ok[j]) {
                    mw[slot_head[j]] = m2[j];
                    mw[G + slot_head[j]] = l2[j];
                }
        }
        named_barrier_sync(1, W * 32);
        if (threadIdx.x == 0) *stop_flag = *abort_flag;
        named_barrier_sync(1, W * 32);
        if (*stop_flag) {
            // some wait of this CTA gave up: the item is abandoned
            ok = false;
            abandon_rows(r);
            continue;
        }

        // ---- CTA merge of the warps' partial states
        const int64_t split0 = int64_t(r.s) * a.batch * T * a.num_q_heads;
        for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
            const int head = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, merge[w * (2 * G + G * D) + head]);
            float out = 0.f, lsum = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float *mwx = merge + w * (2 * G + G * D);
                    const float wt = exp2f(mwx[head] - M);
                    lsum = fmaf(wt, mwx[G + head], lsum);
                    out = fmaf(wt, mwx[2 * G + head * D + d], out);
                }
                out /= lsum;
            }
            const int64_t orow = split0 + row_offset(a, r.b, r.g, head, Gr);
            a.out_part[orow * D + d] = out;
            if (d == 0) a.lse_part[orow] = M != -INFINITY ? (M + log2f(lsum)) * kLn2 : -INFINITY;
        }
        named_barrier_sync(1, W * 32);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// The pool as rows of `dim` bf16.  D = 128: a 3-D map (64 columns, rows,
// 2 halves at a 128-byte stride) whose box -- one segment of rows, both
// halves -- reads one contiguous run of HBM and lands half-major; D = 64: a
// 2-D map (64 columns, rows).
bool make_pool_map(CUtensorMap *map, const void *pool, int64_t rows, int dim, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t rank = dim == 128 ? 3 : 2;
    cuuint64_t gdim[3] = {64, cuuint64_t(rows), 2};
    cuuint64_t gstride[2] = {cuuint64_t(dim) * 2, 128};
    cuuint32_t box[3] = {64, cuuint32_t(box_rows), 2};
    cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(pool), gdim, gstride,
              box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs of this instance the current device keeps resident per SM (the
// occupancy the launch's persistent grid is sized by; the split-count model
// uses the same figure).  Sets the kernel's shared-memory attribute first.
// Cached per device and thread; 0 if the runtime failed.
template <int D, int G, int W, int NSTAGES, int MINB>
int resident_per_sm() {
    using C = Cfg<D, G, W, NSTAGES, MINB>;
    auto kernel = decode_tma_kernel<D, G, W, NSTAGES, MINB>;
    static thread_local int configured_dev = -1, cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (configured_dev != dev) {
        int per_sm = 0;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(C::kSmemBytes)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, C::kThreads,
                                                          C::kSmemBytes) != cudaSuccess)
            return 0;
        cached = per_sm;
        configured_dev = dev;
    }
    return cached;
}

template <int D, int G, int W, int NSTAGES, int MINB>
int launch(const DecodeArgs &a) {
    using C = Cfg<D, G, W, NSTAGES, MINB>;
    auto kernel = decode_tma_kernel<D, G, W, NSTAGES, MINB>;
    const int64_t rows = int64_t(a.cache.num_blocks) * a.cache.num_kv_heads * a.cache.block_size;
    const int box_rows = std::min(a.cache.block_size, C::kStageTokens);
    CUtensorMap tk, tv;
    if (!make_pool_map(&tk, a.k_pool, rows, D, box_rows) ||
        !make_pool_map(&tv, a.v_pool, rows, D, box_rows))
        return PKV_ERR_CUDA;
    const int per_sm = resident_per_sm<D, G, W, NSTAGES, MINB>();
    if (per_sm < 1) return PKV_ERR_CUDA;
    const int64_t items = int64_t(a.batch) * a.cache.num_kv_heads * a.num_splits;
    const int grid = int(std::min<int64_t>(items, int64_t(sm_count()) * per_sm));
    if (grid <= 0) return PKV_OK;
    return launch_pdl(kernel, dim3(grid), dim3(C::kThreads), C::kSmemBytes, a.stream, tk, tv, a);
}

// Launch shapes: consumer warps (W), stages (S), CTAs per SM (B).
#ifndef PKV_TMA_D128_W
#define PKV_TMA_D128_W 2
#endif
#ifndef PKV_TMA_D128_S
#define PKV_TMA_D128_S 3
#endif
#ifndef PKV_TMA_D128_B
#define PKV_TMA_D128_B 4
#endif
#ifndef PKV_TMA_D128G8_W
#define PKV_TMA_D128G8_W 2
#endif
#ifndef PKV_TMA_D128G8_S
#define PKV_TMA_D128G8_S 2
#endif
#ifndef PKV_TMA_D128G8_B
#define PKV_TMA_D128G8_B 4
#endif
#ifndef PKV_TMA_D128G16_W
#define PKV_TMA_D128G16_W 4
#endif
#ifndef PKV_TMA_D128G16_S
#define PKV_TMA_D128G16_S 4
#endif
#ifndef PKV_TMA_D128G16_B
#define PKV_TMA_D128G16_B 1
#endif
#ifndef PKV_TMA_D64G16_W
#define PKV_TMA_D64G16_W 2
#endif
#ifndef PKV_TMA_D64G16_S
#define PKV_TMA_D64G16_S 6
#endif
#ifndef PKV_TMA_D64G16_B
#define PKV_TMA_D64G16_B 2
#endif
#ifndef PKV_TMA_D64_W
#define PKV_TMA_D64_W 2
#endif
#ifndef PKV_TMA_D64_S
#define PKV_TMA_D64_S 6
#endif
#ifndef PKV_TMA_D64_B
#define PKV_TMA_D64_B 4
#endif
#define PKV_TMA_SHAPE_D128 PKV_TMA_D128_W, PKV_TMA_D128_S, PKV_TMA_D128_B
#define PKV_TMA_SHAPE_D128_G8 PKV_TMA_D128G8_W, PKV_TMA_D128G8_S, PKV_TMA_D128G8_B
#define PKV_TMA_SHAPE_D128_G16 PKV_TMA_D128G16_W, PKV_TMA_D128G16_S, PKV_TMA_D128G16_B
#define PKV_TMA_SHAPE_D64 PKV_TMA_D64_W, PKV_TMA_D64_S, PKV_TMA_D64_B
#define PKV_TMA_SHAPE_D64_G16 PKV_TMA_D64G16_W, PKV_TMA_D64G16_S, PKV_TMA_D64G16_B

}  // namespace

bool tma_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads, int32_t q_tokens) {
    const int G = num_q_heads / c.num_kv_heads * q_tokens;     // query rows per work item
    const bool pow2_bs = c.block_size >= 8 && c.block_size <= 256 &&
                         (c.block_size & (c.block_size - 1)) == 0;
    const int64_t rows = int64_t(c.num_blocks) * c.num_kv_heads * c.block_size;
    return c.head_dim_k == c.head_dim_v && (c.head_dim_k == 64 || c.head_dim_k == 128) &&
           (G == 1 || G == 2 || G == 4 || G == 8 || G == 16) && pow2_bs &&
           rows < (int64_t(1) << 31) - 1;
}

// Launch shapes (consumer warps, stages, CTAs per SM), measured on 8 x 32K
// GQA decode: two consumer warps per CTA (32-token stages) and four CTAs per
// SM keep more independent warps streaming than one large CTA does (G <= 4:
// three stages; G = 8, whose registers leave room for only two stages at
// four CTAs per SM: two).  G = 16 holds twice G = 8's accumulators and does
// four times G = 4's warp-level MMAs per byte: one CTA of four consumer warps
// and four stages per SM was fastest (8 x 32K, 128/8 heads: 300 us against
// 361 us for two 2-warp CTAs and 513-570 us for three CTAs per SM).
int tma_resident_ctas(const pkv_cache_desc &c, int32_t num_q_heads, int32_t q_tokens) {
    const int G = num_q_heads / c.num_kv_heads * q_tokens;
    int per_sm = 0;
    if (c.head_dim_k == 128) {
        switch (G) {
            case 1: per_sm = resident_per_sm<128, 1, PKV_TMA_SHAPE_D128>(); break;
            case 2: per_sm = resident_per_sm<128, 2, PKV_TMA_SHAPE_D128>(); break;
            case 4: per_sm = resident_per_sm<128, 4, PKV_TMA_SHAPE_D128>(); break;
            case 8: per_sm = resident_per_sm<128, 8, PKV_TMA_SHAPE_D128_G8>(); break;
            case 16: per_sm = resident_per_sm<128, 16, PKV_TMA_SHAPE_D128_G16>(); break;
            default: break;
        }
    } else {
        switch (G) {
            case 1: per_sm = resident_per_sm<64, 1, PKV_TMA_SHAPE_D64>(); break;
            case 2: per_sm = resident_per_sm<64, 2, PKV_TMA_SHAPE_D64>(); break;
            case 4: per_sm = resident_per_sm<64, 4, PKV_TMA_SHAPE_D64>(); break;
            case 8: per_sm = resident_per_sm<64, 8, PKV_TMA_SHAPE_D64>(); break;
            case 16: per_sm = resident_per_sm<64, 16, PKV_TMA_SHAPE_D64_G16>(); break;
            default: break;
        }
    }
    return sm_count() * std::max(per_sm, 1);
}

int launch_decode_tma(const DecodeArgs &a) {
    const int G = a.num_q_heads / a.cache.num_kv_heads * a.q_tokens;   // rows per work item
    if (a.cache.head_dim_k == 128) {
        switch (G) {
            case 1: return launch<128, 1, PKV_TMA_SHAPE_D128>(a);
            case 2: return launch<128, 2, PKV_TMA_SHAPE_D128>(a);
            case 4: return launch<128, 4, PKV_TMA_SHAPE_D128>(a);
            case 8: return launch<128, 8, PKV_TMA_SHAPE_D128_G8>(a);
            case 16: return launch<128, 16, PKV_TMA_SHAPE_D128_G16>(a);
            default: return PKV_ERR_SHAPE;
        }
    }
    switch (G) {
        case 1: return launch<64, 1, PKV_TMA_SHAPE_D64>(a);
        case 2: return launch<64, 2, PKV_TMA_SHAPE_D64>(a);
        case 4: return launch<64, 4, PKV_TMA_SHAPE_D64>(a);
        case 8: return launch<64, 8, PKV_TMA_SHAPE_D64>(a);
        case 16: return launch<64, 16, PKV_TMA_SHAPE_D64_G16>(a);
        default: return PKV_ERR_SHAPE;
    }
}

}  // namespace pkv
