// decode_gqa_tc_e4m3.cu -- paged decode attention over an FP8 (E4M3) cache
// with per-KV-head scales, for query groups of R = 4, 8 or 16 heads and head
// dims 128, on the 5th-generation tensor cores of sm_103a with E4M3
// operands (tcgen05.mma kind::f8f6f4, fp32 accumulators in tensor memory).
//
// The cache bytes go to the tensor cores as they are stored.  The fp32
// query cannot: it is carried as four E4M3 terms per element, y = t0 +
// t1/16 + t2/256 + t3/4096 with y = q * scale * log2(e) * k_scale / s_h
// (s_h a power of two putting row h's largest element in [128, 256)), each
// term the E4M3 rounding of the previous residual times 16.  Likewise each
// probability p in [0, 2^8] becomes five terms.  So the score and value
// products keep ~16 significant bits of both, as the bf16 hi/lo split of
// the other kernels does, and the terms ride in the MMA's N:
//   S^T[128 tok x 4R]   = K_tile . Qterms^T          (M=128, N=4R,  K=32)
//   O^T[128 dv x NP]   += V_tile^T . Pterms^T        (M=128, N=NP,  K=32)
// (NP = 5R rounded up to a multiple of 16; the pad rows of P stay zero).
// Column k*R + h holds term k of row h; the softmax and the epilogue fold
// the terms back with weights 16^-k.
//
// Work item = (sequence b, KV head g, split chunk s), walked in 128-token
// tiles; a tile of K (or V) is 128 rows of 128 bytes, one 16 KB ring stage,
// each KV block one TMA box (issued by one lane of the producer warp).
// Warp roles as in the bf16 tcgen05 GQA kernel: warp 0 TMA producer, warp 1
// TMEM owner and MMA issuer (it also zeroes value rows past a sequence's
// end), warps 2-5 one thread per token lane for the query split, the
// stale-max online softmax (the running max rises only past a slack of 8 in
// log2 units; the accumulators are then rescaled in TMEM) and the
// epilogue.  Groups of 16 run two CTAs per SM (~111 KB of shared memory
// each), groups of 4 and 8 three.  Every wait is bounded.
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

// Groups of 4 and 8: small operand arrays, so three CTAs per SM with three
// ring stages each (measured on 8 x 32K: 89.8 us against 96.5 us for two
// CTAs with five stages at groups of 4; 97.4 us against 102.5 us at groups
// of 8, whose registers then go from 121 to 96 with a 24-byte spill).
// Groups of 8 on two CTAs with two softmax groups (SG 2, probabilities
// MN-major) matched three CTAs per DCP step but did not beat it.
#ifndef PKV_E4M3_R4_RING
#define PKV_E4M3_R4_RING 3
#endif
#ifndef PKV_E4M3_R4_CTAS
#define PKV_E4M3_R4_CTAS 3
#endif
#ifndef PKV_E4M3_R8_RING
#define PKV_E4M3_R8_RING 3
#endif
#ifndef PKV_E4M3_R8_CTAS
#define PKV_E4M3_R8_CTAS 3
#endif
#ifndef PKV_E4M3_R8_SG
#define PKV_E4M3_R8_SG 1
#endif
// Groups of 16: two CTAs per SM, each with two softmax warp groups of four
// warps (8 rows each) and the probabilities MN-major (a token's terms stored
// with one 16-byte store per term half) -- the 16-row softmax was bound by
// its own instruction chain per warp -- and five ring stages beside one
// probability buffer (108.9 us per speculative step against 111.2 us with
// four stages and two buffers).
#ifndef PKV_E4M3_R16_SG
#define PKV_E4M3_R16_SG 2
#endif
#ifndef PKV_E4M3_R16_RING
#define PKV_E4M3_R16_RING 5
#endif
// Probability buffers (1 or 2) per form: one buffer frees its bytes for a
// ring stage, the softmax then writes tile i + 1's terms after the value
// product of tile i.
#ifndef PKV_E4M3_R4_PBUF
#define PKV_E4M3_R4_PBUF 2
#endif
#ifndef PKV_E4M3_R8_PBUF
#define PKV_E4M3_R8_PBUF 2
#endif
#ifndef PKV_E4M3_R16_PBUF
#define PKV_E4M3_R16_PBUF 1
#endif

namespace pkv {
namespace {

constexpr int kM = 128;                 // tokens per tile
constexpr int kD = 128;                 // head dim (bytes of an E4M3 row)
constexpr int kStage = kM * kD;         // one K or V tile: 16 KB
constexpr int kSoftWarp0 = 2;
constexpr int kSoftThreads = 128;
constexpr int kQTerms = 4, kPTerms = 5;
// The value product of tile i is issued after the score product of tile
// i + kLag (and the producer loads V of tile i after K of tile i + kLag).
// Measured at 16 rows over 8 x 32K: a lag of two (the score product of tile
// i + 1 no longer queued behind the probabilities of tile i - 1) was no
// faster than one, and slower at 8 rows (value stages held a tile longer).
constexpr int kLag = 1;
constexpr float kSlack = 8.f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Rows R per item, ring stages, CTAs per SM, softmax warp groups SG (each
// of four warps, one thread per token lane, taking R / SG of the rows), the
// probability operand's layout: PMN = MN-major (a token's terms
// contiguous: [128 tokens][128 B], N = 128, so a thread stores its terms
// with one vector store per term), else K-major ([NP rows][128 tokens],
// one byte store per term and row), and the probability buffers NPB.
template <int R, int RING, int CTAS, int SG, bool PMN, int NPB>
struct Cfg {
    static constexpr int kRing = RING;
    static constexpr int kCtas = CTAS;
    static constexpr int kThreads = 64 + 128 * SG;
    static constexpr int kNQ = kQTerms * R;                         // score MMA N
    static constexpr int kNP = PMN ? 128 : (kPTerms * R + 15) / 16 * 16;   // value MMA N
    static constexpr uint32_t kColO = 2 * kNQ;                      // S^T buffers first
    static constexpr uint32_t kTmemCols =
        2 * kNQ + kNP <= 64 ? 64 : 2 * kNQ + kNP <= 128 ? 128 : 256;
    static constexpr uint32_t kPBytes = kNP * 128;                  // one probability buffer
    // Shared memory after the 1024-byte misc block: the query terms
    // [4R rows][128 B], NPB probability buffers [NP rows][128 B], the ring.
    static constexpr uint32_t kOffP = 1024 + kNQ * 128;
    static constexpr uint32_t kOffRing = kOffP + NPB * kPBytes;
    static constexpr uint32_t kSmemBytes = 1024 + kOffRing + RING * kStage;
    static_assert(kOffP % 1024 == 0 && kOffRing % 1024 == 0, "1024-byte-aligned operands");
    static_assert(RING <= 8, "mbarrier slots for at most 8 stages");
    static_assert(NPB == 1 || NPB == 2, "one or two probability buffers");
};

// mbarrier slots
constexpr int kBarFull = 0;             // + stage
constexpr int kBarEmpty = 8;            // + stage
constexpr int kBarSFull = 16;           // + buffer
constexpr int kBarSEmpty = 18;          // + buffer
constexpr int kBarPFull = 20;           // + P buffer
constexpr int kBarPvDone = 22;          // + P buffer
constexpr int kBarQFull = 24;
constexpr int kBarQEmpty = 25;
constexpr int kBarOEmpty = 26;
constexpr int kBarDrain = 27;

// Shared memory, offsets from a 1024-byte-aligned base (the operand arrays
// follow in Cfg).
constexpr uint32_t kOffMrow = 256;                      // running max per row (log2)
constexpr uint32_t kOffAux = kOffMrow + 64;             // rescale factor, then 1/l
constexpr uint32_t kOffQsc = kOffAux + 64;              // power-of-two scale s_h of row h
constexpr uint32_t kOffRed = kOffQsc + 64;              // [4 warps][16 rows]
constexpr uint32_t kOffSlot = kOffRed + 256;
constexpr uint32_t kOffFlag = kOffSlot + 4;
constexpr uint32_t kOffQ = 1024;

__device__ __forceinline__ int64_t lmin(int64_t x, int64_t y) { return x < y ? x : y; }

// The next terms' inputs after the E4M3 codes c (bits 0-7: x0's, 8-15:
// x1's): x_i <- 16 (x_i - v_i), v_i the value of code i, as one
// mixed-precision fma per element on v_i in fp16 (every E4M3 value is an
// fp16 value): 16 x_i - 16 v_i.  v_i is x_i rounded to four significant
// bits, so the difference, its product by 16 and hence the single rounding
// of the fma are exact -- the same bits as a subtraction then a product.
__device__ __forceinline__ void residual16(uint32_t c, float &x0, float &x1) {
    uint32_t h2;
    asm("{ .reg .b16 c; cvt.u16.u32 c, %1; cvt.rn.f16x2.e4m3x2 %0, c; }" : "=r"(h2) : "r"(c));
    const float a0 = 16.f * x0, a1 = 16.f * x1;
    asm("{ .reg .b16 l, h, m; mov.b16 m, 0xCC00; mov.b32 {l, h}, %2; "
        "fma.rn.f32.f16 %0, l, m, %3; fma.rn.f32.f16 %1, h, m, %4; }"   // m = -16
        : "=f"(x0), "=f"(x1) : "r"(h2), "f"(a0), "f"(a1));
}

// Byte offset of (row, column < 128) in a [rows][128 B] array with the
// 128-byte swizzle (8-row atoms 1024-byte aligned).
__device__ __forceinline__ uint32_t swz8(int row, int col) {
    return uint32_t(row) * 128 + (uint32_t(((col >> 4) ^ row) & 7) << 4) + uint32_t(col & 15);
}

struct Item {
    int b, g, s, hg;
    int64_t len, begin, end;
    int ntiles;
};

// Head groups of R rows per (sequence, KV head): 1, or 2 for a 32-row group
// (G x T = 32) taken as two items of 16.
template <int R>
__device__ __forceinline__ int head_groups(const DecodeArgs &a) {
    if constexpr (R < 16) return 1;   // 4 and 8 rows: the whole group
    else return a.num_q_heads / a.cache.num_kv_heads * a.q_tokens / R;
}

// item = ((b * Hkv + g) * S + s) * HG + hg, the head group fastest (the two
// groups of a chunk read the same tiles together).  Split s of (b, g) covers
// tokens [s C, min(L, (s + 1) C)), C = 64 ceil(L / 64 S).
__device__ __forceinline__ Item fp8_item(const DecodeArgs &a, int item, int HG, bool report) {
    Item r;
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

template <int R, int RING, int CTAS, int SG, bool PMN, int NPB>
__global__ void __launch_bounds__(64 + 128 * SG, CTAS)
decode_gqa_tc_e4m3_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
    using S = Cfg<R, RING, CTAS, SG, PMN, NPB>;
    constexpr int kRing = RING;
    constexpr uint32_t kOffP = S::kOffP, kOffRing = S::kOffRing;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(base);
    float *mrow = reinterpret_cast<float *>(base + kOffMrow);
    float *aux = reinterpret_cast<float *>(base + kOffAux);
    float *qsc = reinterpret_cast<float *>(base + kOffQsc);
    float *red = reinterpret_cast<float *>(base + kOffRed);
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(base + kOffSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kOffFlag);
    auto bar = [&](int i) { return sb + 8u * uint32_t(i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_items = a.batch * a.cache.num_kv_heads * a.num_splits * head_groups<R>(a);
    const int bs = a.cache.block_size, hkv = a.cache.num_kv_heads;
    const int box = bs < kM ? bs : kM;                 // rows per TMA box (one block or less)

    if (threadIdx.x == 0) {
        for (int r = 0; r < kRing; ++r) {
            mbar_init(bar(kBarFull + r), 1);
            mbar_init(bar(kBarEmpty + r), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarSFull + i), 1);
            mbar_init(bar(kBarSEmpty + i), kSoftThreads * SG);
            mbar_init(bar(kBarPFull + i), kSoftThreads * SG);
            mbar_init(bar(kBarPvDone + i), 1);
        }
        mbar_init(bar(kBarQFull), kSoftThreads * SG);
        mbar_init(bar(kBarQEmpty), 1);
        mbar_init(bar(kBarOEmpty), kSoftThreads * SG);
        mbar_init(bar(kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::alloc(sb + kOffSlot, S::kTmemCols);
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
        const int nbox = kM / box;                     // boxes per tile (<= 8)
        for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
            const Item r = fp8_item(a, item, head_groups<R>(a), false);
            if (r.ntiles == 0) continue;
            const int32_t *table = a.block_tables + int64_t(r.b) * a.max_blocks;
            // Rows of block 0 of this KV head stand in for boxes past the end
            // (masked scores, zeroed value rows).
            const int32_t standin = r.g * bs;
            int32_t ylag[kLag];                        // rows of tiles i - 1, i - 2
#pragma unroll
            for (int l = 0; l < kLag; ++l) ylag[l] = standin;
            // One table read resolves the boxes of tpg tiles (lane j: box
            // j % nbox of tile j / nbox of the group); the next group's
            // entries are loaded a group ahead, so no table read waits in
            // front of a copy.
            const int tpg = 32 / nbox;
            auto first_token = [&](int i0) -> int64_t {   // of this lane's box, or -1
                const int ti = i0 + lane / nbox;
                const int64_t t = r.begin + int64_t(ti) * kM + int64_t(lane % nbox) * box;
                return ti < r.ntiles && t < r.end ? t : -1;
            };
            auto fetch = [&](int i0) -> int32_t {
                const int64_t t = first_token(i0);
                return t >= 0 ? table[t / bs] : 0;
            };
            int32_t phys_next = fetch(0);
            int32_t yg = standin;
            for (int i = 0; i < r.ntiles + kLag && ok; ++i) {
                if (i % tpg == 0) {
                    const int32_t phys = phys_next;
                    phys_next = fetch(i + tpg);
                    const int64_t t = first_token(i);
                    yg = standin;
                    if (t >= 0) {
                        if (phys >= 0 && phys < a.cache.num_blocks)
                            yg = (phys * hkv + r.g) * bs + int32_t(t % bs);
                        else
                            raise_status(a.status, PKV_DEV_BLOCK_ID);
                    }
                }
                // lane j < nbox: row of box j of tile i
                const int32_t y = __shfl_sync(0xffffffffu, yg, (i % tpg) * nbox + lane % nbox);
                // K of tile i, then V of tile i - kLag: one stage each
                for (int kv = (i < r.ntiles ? 0 : 1); kv < (i >= kLag ? 2 : 1); ++kv) {
                    const bool w = pipe_wait(bar(kBarEmpty + stage), phase ^ 1u, a.status,
                                             abort_flag);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(bar(kBarFull + stage), kStage);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    __syncwarp();
                    if (lane < nbox)
                        tma_load_2d(sb + kOffRing + uint32_t(stage) * kStage +
                                        uint32_t(lane * box) * kD,
                                    kv == 0 ? &tmap_k : &tmap_v, 0, kv == 0 ? y : ylag[kLag - 1],
                                    bar(kBarFull + stage));
                    if (++stage == kRing) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
#pragma unroll
                for (int l = kLag - 1; l > 0; --l) ylag[l] = ylag[l - 1];
                ylag[0] = y;
            }
        }
        // leave no copy in flight into this CTA's shared memory
        if (lane == 0)
            for (int s = 0; s < kRing; ++s)
                if (armed & (1u << s))
                    mbar_wait(bar(kBarFull + s), (armed_parity >> s) & 1u, a.status);
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdS = tc::idesc_e4m3_f32(128, S::kNQ, 0, 0);   // K-major K, K-major Q
        // MN-major V; P K-major, or MN-major when PMN
        constexpr uint32_t kIdO = tc::idesc_e4m3_f32(128, S::kNP, 1, PMN ? 1 : 0);
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
            const Item r = fp8_item(a, item, head_groups<R>(a), false);
            if (r.ntiles == 0) continue;
            if (!(ok = wait_all(bar(kBarQFull), ne & 1u))) break;
            for (int i = 0; i < r.ntiles + kLag && ok; ++i) {
                if (i < r.ntiles) {
                    // ---- S^T[buf] = K_tile . Qterms^T
                    const uint32_t buf = tcount & 1u;
                    if (!(ok = wait_all(bar(kBarSEmpty + buf), ((tcount >> 1) & 1u) ^ 1u))) break;
                    if (!(ok = wait_all(bar(kBarFull + stage), phase))) break;
                    tc::fence_after_sync();
                    if (lane == 0) {
                        const uint32_t kb = sb + kOffRing + uint32_t(stage) * kStage;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_e4m3(tmem + S::kNQ * buf, tc::smem_desc(kb + 32 * kk, 16, 1024),
                                         tc::smem_desc(qb + 32 * kk, 16, 1024), kIdS, kk != 0);
                        tc::commit(bar(kBarEmpty + stage));
                        tc::commit(bar(kBarSFull + buf));
                        if (i == r.ntiles - 1) tc::commit(bar(kBarQEmpty));
                    }
                    __syncwarp();
                    advance();
                    ++tcount;
                }
                if (i >= kLag) {
                    // ---- O^T += V_tile^T . Pterms^T for tile j
                    const int j = i - kLag;
                    const uint32_t pbuf = pcount % NPB;
                    if (!(ok = wait_all(bar(kBarPFull + pbuf), (pcount / NPB) & 1u))) break;
                    if (j == 0 && !(ok = wait_all(bar(kBarOEmpty), (ne & 1u) ^ 1u))) break;
                    if (!(ok = wait_all(bar(kBarFull + stage), phase))) break;
                    const int64_t tok0 = r.begin + int64_t(j) * kM;
                    const int nvalid = int(lmin(kM, r.end - tok0));
                    if (nvalid < kM) {
                        // value rows past the end may hold any bits (NaN
                        // times a zero probability is NaN): zero them
                        uint8_t *vt = base + kOffRing + size_t(stage) * kStage;
                        for (int idx = lane; idx < (kM - nvalid) * 8; idx += 32)
                            *reinterpret_cast<uint4 *>(vt + (nvalid + (idx >> 3)) * kD +
                                                       (idx & 7) * 16) = make_uint4(0, 0, 0, 0);
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    tc::fence_after_sync();
                    if (lane == 0) {
                        const uint32_t vb = sb + kOffRing + uint32_t(stage) * kStage;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // 32 tokens a step: 32 rows of the MN-major layouts,
                            // 32 bytes along a K-major row
                            const uint32_t pa = pb + pbuf * S::kPBytes;
                            tc::mma_e4m3(tmem + S::kColO,
                                         tc::smem_desc(vb + 4096 * kk, 16384, 1024),
                                         PMN ? tc::smem_desc(pa + 4096 * kk, 16384, 1024)
                                             : tc::smem_desc(pa + 32 * kk, 16, 1024),
                                         kIdO, (j | kk) != 0);
                        }
                        tc::commit(bar(kBarEmpty + stage));
                        tc::commit(bar(kBarPvDone + pbuf));
                    }
                    __syncwarp();
                    advance();
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
        // SG groups of four warps; group grp takes rows h0 .. h0 + RG - 1, each
        // thread one token lane (S^T) / value row (O^T) of its quadrant.
        constexpr int RG = R / SG;
        const int grp = (warp - kSoftWarp0) >> 2;
        const int tt = threadIdx.x - kSoftWarp0 * 32;            // 0 .. 128 SG - 1
        const int t = tt - 128 * grp;                              // 0..127 within the group
        const int h0 = grp * RG;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;                // token lane of S^T, value row of O^T
        const uint32_t tl = tmem + (uint32_t(quad * 32) << 16);
        uint8_t *qs = base + kOffQ, *ps = base + kOffP;
        constexpr int kTpr = 128 * SG / R;               // threads per query row in the split
        constexpr int kDpt = kD / kTpr;                  // query dims per thread
        uint32_t tcount = 0, pcount = 0, ne = 0;
        // the pad rows (columns) of the probability buffers stay zero
        for (int i = tt; i < NPB * int(S::kPBytes) / 16; i += kSoftThreads * SG)
            reinterpret_cast<uint4 *>(ps)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        auto wait_pv = [&](uint32_t j) {
            return pipe_wait(bar(kBarPvDone + j % NPB), (j / NPB) & 1u, a.status, abort_flag);
        };
        // barrier 1 + grp over this group's 128 threads (an OR of `pred`)
        auto gbar_or = [&](bool pred) -> bool {
            uint32_t v;
            asm volatile(
                "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, 128, p; "
                "selp.u32 %0, 1, 0, q; }"
                : "=r"(v) : "r"(uint32_t(pred)), "r"(1 + grp) : "memory");
            return v != 0;
        };
        auto gbar = [&]() { named_barrier_sync(1 + uint32_t(grp), 128); };
        // The R rows of an item are T query tokens x Gr heads: row h is query
        // token h / Gr of sequence b, head g G + hg Gr + h % Gr (T = 1, one
        // head group: the group).
        // (T, Gr and the shift are re-read from the parameters where used:
        // kept live across the tile loop they cost registers)
        auto gr_shift = [&]() { return __ffs(R / a.q_tokens) - 1; };
        for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
            const Item r = fp8_item(a, item, head_groups<R>(a), tt == 0);
            auto row_of = [&](int h) -> int64_t {
                const int sh = gr_shift(), Gr = R / a.q_tokens;
                const int G = a.num_q_heads / a.cache.num_kv_heads;
                return (int64_t(r.b) * a.q_tokens + (h >> sh)) * a.num_q_heads +
                       int64_t(r.g) * G + r.hg * Gr + (h & (Gr - 1));
            };
            const int64_t split0 = int64_t(r.s) * a.batch * a.q_tokens * a.num_q_heads;
            if (r.ntiles == 0) {
                for (int i = tt; i < R * kD / 4; i += kSoftThreads * SG)
                    reinterpret_cast<float4 *>(a.out_part + (split0 + row_of(i / (kD / 4))) *
                                                                kD)[i % (kD / 4)] =
                        make_float4(0.f, 0.f, 0.f, 0.f);
                if (tt < R) a.lse_part[split0 + row_of(tt)] = -INFINITY;
                continue;
            }
            // ---- the item's query rows as four E4M3 terms each (rows k R + h
            // of the score MMA's K-major B operand); thread tt holds kDpt dims
            // of row tt / kTpr (a row of this thread's own group)
            bool w = pipe_wait(bar(kBarQEmpty), (ne & 1u) ^ 1u, a.status, abort_flag);
            if (w) {
                const int h = tt / kTpr, d0 = (tt % kTpr) * kDpt;
                const float qmul = a.scale * kLog2e * a.k_scale[r.g];
                const float4 *src = reinterpret_cast<const float4 *>(a.q + row_of(h) * kD + d0);
                float x[kDpt];
                float amax = 0.f;
#pragma unroll
                for (int v = 0; v < kDpt / 4; ++v) {
                    const float4 f = src[v];
                    x[4 * v] = f.x * qmul;
                    x[4 * v + 1] = f.y * qmul;
                    x[4 * v + 2] = f.z * qmul;
                    x[4 * v + 3] = f.w * qmul;
                }
#pragma unroll
                for (int e = 0; e < kDpt; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
                for (int o = kTpr / 2; o > 0; o >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                // s_h = 2^(floor(log2 max|x|) - 7): the row's largest term-0
                // magnitude lies in [128, 256), below E4M3's 448
                const int e2 = amax > 0.f ? max(ilogbf(amax), -110) : 0;
                const float inv = ldexpf(1.f, 7 - e2);
                if (tt % kTpr == 0) qsc[h] = ldexpf(1.f, e2 - 7);
#pragma unroll
                for (int e = 0; e < kDpt; ++e) x[e] *= inv;
#pragma unroll
                for (int k = 0; k < kQTerms; ++k)
#pragma unroll
                    for (int e = 0; e < kDpt; e += 4) {
                        const uint32_t c01 = e4m3x2_from_f32(x[e], x[e + 1]);
                        const uint32_t c23 = e4m3x2_from_f32(x[e + 2], x[e + 3]);
                        *reinterpret_cast<uint32_t *>(qs + swz8(k * R + h, d0 + e)) =
                            c01 | (c23 << 16);
                        residual16(c01, x[e], x[e + 1]);
                        residual16(c23, x[e + 2], x[e + 3]);
                    }
                fence_proxy_async_smem();
            }
            mbar_arrive(bar(kBarQFull));
            if (t < RG) mrow[h0 + t] = -INFINITY;
            float l_part[RG];
#pragma unroll
            for (int j = 0; j < RG; ++j) l_part[j] = 0.f;
            const int32_t span = int32_t(r.end - r.begin);
            // causal limits, from r.begin: row h sees tokens < lim0 + h / Gr
            const int32_t lim0 = int32_t(r.len - (a.q_tokens - 1) - r.begin);
            if (gbar_or(!w)) break;          // also orders qsc and mrow in the group

            bool ok = true;
            for (int i = 0; i < r.ntiles; ++i) {
                const uint32_t buf = tcount & 1u;
                w = pipe_wait(bar(kBarSFull + buf), (tcount >> 1) & 1u, a.status, abort_flag);
                float x[RG];
                {
                    uint32_t v[kQTerms][RG];
                    tc::fence_after_sync();
#pragma unroll
                    for (int k = 0; k < kQTerms; ++k)
                        tc::ldn<RG>(tl + S::kNQ * buf + k * R + h0, v[k]);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < RG; ++j) {      // fold the query terms back
                        float s = __uint_as_float(v[kQTerms - 1][j]);
#pragma unroll
                        for (int k = kQTerms - 2; k >= 0; --k)
                            s = fmaf(s, 0.0625f, __uint_as_float(v[k][j]));
                        x[j] = s * qsc[h0 + j];
                    }
                }
                tc::fence_before_sync();
                mbar_arrive(bar(kBarSEmpty + buf));
                ++tcount;
                // this token is seen by rows h >= hmin (none past the span)
                const int32_t tok = i * kM + row, rel = tok - lim0;   // from r.begin
                const int hmin =
                    tok >= span ? R : rel < 0 ? 0 : min(rel + 1, a.q_tokens) << gr_shift();
                bool need = false;
#pragma unroll
                for (int j = 0; j < RG; ++j) {
                    x[j] = h0 + j >= hmin ? x[j] : -INFINITY;
                    need |= x[j] > mrow[h0 + j] + kSlack;
                }
                // one group barrier in the common case (no failed wait, no
                // rise of a running max); the rare cases are told apart after it
                bool rise = false;
                if (gbar_or(need || !w)) {
                    if (gbar_or(!w)) {
                        ok = false;
                        break;
                    }
                    rise = gbar_or(need);
                }
                if (rise) {
#pragma unroll
                    for (int j = 0; j < RG; ++j) {
                        float m = x[j];
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                        if (lane == j) red[quad * 16 + h0 + j] = m;
                    }
                    gbar();
                    if (t < RG) {
                        const int h = h0 + t;
                        const float tm = fmaxf(fmaxf(red[h], red[16 + h]),
                                               fmaxf(red[32 + h], red[48 + h]));
                        const float mo = mrow[h], mn = fmaxf(mo, tm);
                        aux[h] = (mo == -INFINITY || mn == -INFINITY) ? 0.f : exp2f(mo - mn);
                        mrow[h] = mn;
                    }
                    gbar();
#pragma unroll
                    for (int j = 0; j < RG; ++j) l_part[j] *= aux[h0 + j];
                    if (i > 0) {
                        // the accumulators are quiet once the previous tile's
                        // value MMAs are done: rescale this group's columns
                        const bool wv = wait_pv(pcount - 1);
                        tc::fence_after_sync();
                        if (wv) {
#pragma unroll
                            for (int k = 0; k < kPTerms; ++k) {
                                uint32_t v[RG];
                                const uint32_t ta = tl + S::kColO + k * R + h0;
                                tc::ldn<RG>(ta, v);
                                tc::wait_ld();
#pragma unroll
                                for (int j = 0; j < RG; ++j)
                                    v[j] = __float_as_uint(__uint_as_float(v[j]) * aux[h0 + j]);
                                tc::stn<RG>(ta, v);
                            }
                            tc::wait_st();
                        }
                    }
                }
                float p[RG];
#pragma unroll
                for (int j = 0; j < RG; ++j) {
                    p[j] = x[j] == -INFINITY ? 0.f : ex2_approx(x[j] - mrow[h0 + j]);
                    l_part[j] += p[j];
                }
                // this P buffer was last read by the value MMAs of tile
                // pcount - NPB
                if (pcount >= NPB) wait_pv(pcount - NPB);
                {
                    // five E4M3 terms of each probability (p <= 2^8): term k of
                    // row h is column k R + h of the value MMA's B operand,
                    // this thread's token its row (MN-major) or its column
                    uint8_t *pa = ps + (pcount % NPB) * S::kPBytes;
#pragma unroll
                    for (int k = 0; k < kPTerms; ++k) {
                        uint32_t word[(RG + 3) / 4];
#pragma unroll
                        for (int j = 0; j < RG; j += 2) {
                            const uint32_t c = e4m3x2_from_f32(p[j], p[j + 1]);
                            if constexpr (PMN) {
                                if ((j & 3) == 0) word[j >> 2] = c;
                                else word[j >> 2] |= c << 16;
                            } else {
                                pa[swz8(k * R + h0 + j, row)] = uint8_t(c);
                                pa[swz8(k * R + h0 + j + 1, row)] = uint8_t(c >> 8);
                            }
                            if (k + 1 < kPTerms) residual16(c, p[j], p[j + 1]);
                        }
                        if constexpr (PMN) {
                            // bytes k R + h0 .. + RG of this token's 128-byte row:
                            // inside one 16-byte chunk (RG divides 16)
                            const int n0 = k * R + h0;
                            uint8_t *dst = pa + row * 128 + (((n0 >> 4) ^ (row & 7)) << 4) +
                                           (n0 & 15);
                            if constexpr (RG == 16)
                                *reinterpret_cast<uint4 *>(dst) =
                                    make_uint4(word[0], word[1], word[2], word[3]);
                            else if constexpr (RG == 8)
                                *reinterpret_cast<uint2 *>(dst) = make_uint2(word[0], word[1]);
                            else
                                *reinterpret_cast<uint32_t *>(dst) = word[0];
                        }
                    }
                }
                fence_proxy_async_smem();
                tc::fence_before_sync();
                mbar_arrive(bar(kBarPFull + pcount % NPB));
                ++pcount;
            }
            if (!ok) break;

            // ---- epilogue: the item's last value MMAs are done
            w = wait_pv(pcount - 1);
            tc::fence_after_sync();
#pragma unroll
            for (int j = 0; j < RG; ++j) {
                float s = l_part[j];
                s += __shfl_xor_sync(0xffffffffu, s, 16);
                s += __shfl_xor_sync(0xffffffffu, s, 8);
                s += __shfl_xor_sync(0xffffffffu, s, 4);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                if (lane == j) red[quad * 16 + h0 + j] = s;
            }
            gbar();
            if (t < RG) {
                const int h = h0 + t;
                const float l = (red[h] + red[16 + h]) + (red[32 + h] + red[48 + h]);
                aux[h] = l > 0.f ? a.v_scale[r.g] / l : 0.f;
                a.lse_part[split0 + row_of(h)] = l > 0.f ? (mrow[h] + log2f(l)) * kLn2 : -INFINITY;
            }
            gbar();
            if (w) {
                uint32_t v[kPTerms][RG];
#pragma unroll
                for (int k = 0; k < kPTerms; ++k) tc::ldn<RG>(tl + S::kColO + k * R + h0, v[k]);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < RG; ++j) {          // fold the probability terms back
                    float o = __uint_as_float(v[kPTerms - 1][j]);
#pragma unroll
                    for (int k = kPTerms - 2; k >= 0; --k)
                        o = fmaf(o, 0.0625f, __uint_as_float(v[k][j]));
                    a.out_part[(split0 + row_of(h0 + j)) * kD + row] = o * aux[h0 + j];
                }
            }
            tc::fence_before_sync();
            mbar_arrive(bar(kBarOEmpty));
            ++ne;
            if (gbar_or(!w)) break;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::dealloc(tmem, S::kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 e4m3_encode_fn() {
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

// The pool as rows of 128 one-byte codes; one box = `box` rows, landing as
// [rows][128 B] with the 128-byte swizzle.
bool make_byte_map(CUtensorMap *map, const void *pool, int64_t rows, int box) {
    auto fn = e4m3_encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {cuuint64_t(kD), cuuint64_t(rows)};
    cuuint64_t gstride[1] = {cuuint64_t(kD)};
    cuuint32_t bdim[2] = {cuuint32_t(kD), cuuint32_t(box)};
    cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), gdim, gstride,
              bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int R, int RING, int CTAS, int SG, bool PMN, int NPB>
int launch_rows(const DecodeArgs &a) {
    using S = Cfg<R, RING, CTAS, SG, PMN, NPB>;
    auto kernel = decode_gqa_tc_e4m3_kernel<R, RING, CTAS, SG, PMN, NPB>;
    const int64_t rows = int64_t(a.cache.num_blocks) * a.cache.num_kv_heads * a.cache.block_size;
    const int box = std::min(a.cache.block_size, kM);
    CUtensorMap tk, tv;
    if (!make_byte_map(&tk, a.k_pool, rows, box) || !make_byte_map(&tv, a.v_pool, rows, box))
        return PKV_ERR_CUDA;
    static thread_local int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(S::kSmemBytes)) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_dev = dev;
    }
    // kCtas CTAs per SM by construction (shared memory, registers and TMEM
    // columns are sized for it); the persistent loop is correct for any grid.
    const int64_t items = int64_t(a.batch) * a.cache.num_kv_heads * a.num_splits *
                          (a.num_q_heads / a.cache.num_kv_heads * a.q_tokens / R);
    const int grid = int(std::min<int64_t>(items, int64_t(sm_count()) * CTAS));
    if (grid <= 0) return PKV_OK;
    return launch_pdl(kernel, dim3(grid), dim3(S::kThreads), S::kSmemBytes, a.stream, tk, tv, a);
}

}  // namespace

bool gqa_tc_e4m3_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads,
                                  int32_t q_tokens) {
    if (c.num_kv_heads <= 0 || num_q_heads % c.num_kv_heads != 0 || q_tokens < 1 ||
        q_tokens > 16)
        return false;
    const int G = num_q_heads / c.num_kv_heads * q_tokens;   // rows per item
    const bool pow2_bs = c.block_size >= 16 && c.block_size <= 256 &&
                         (c.block_size & (c.block_size - 1)) == 0;
    const int64_t rows = int64_t(c.num_blocks) * c.num_kv_heads * c.block_size;
    return (G == 4 || G == 8 || G == 16 || G == 32) && c.head_dim_k == kD && c.head_dim_v == kD && pow2_bs &&
           rows < (int64_t(1) << 31) - 1;
}

int gqa_tc_e4m3_head_groups(int32_t group) { return group == 32 ? 2 : 1; }

int gqa_tc_e4m3_resident_ctas(int32_t group) {
    return sm_count() * (group == 4 ? PKV_E4M3_R4_CTAS : group == 8 ? PKV_E4M3_R8_CTAS : 2);
}

int launch_decode_gqa_tc_e4m3(const DecodeArgs &a) {
    switch (a.num_q_heads / a.cache.num_kv_heads * a.q_tokens) {
        case 4:
            return launch_rows<4, PKV_E4M3_R4_RING, PKV_E4M3_R4_CTAS, 1, false, PKV_E4M3_R4_PBUF>(a);
        case 8:
            return launch_rows<8, PKV_E4M3_R8_RING, PKV_E4M3_R8_CTAS, PKV_E4M3_R8_SG,
                               (PKV_E4M3_R8_SG > 1), PKV_E4M3_R8_PBUF>(a);
        case 16:
        case 32:   // 32 rows: two head groups of 16
            return launch_rows<16, PKV_E4M3_R16_RING, 2, PKV_E4M3_R16_SG, (PKV_E4M3_R16_SG > 1),
                               PKV_E4M3_R16_PBUF>(a);
        default: return PKV_ERR_SHAPE;
    }
}

}  // namespace pkv
