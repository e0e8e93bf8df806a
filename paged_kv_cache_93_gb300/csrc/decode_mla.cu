// decode_mla.cu -- paged decode attention for large query groups on sm_103a
// (MLA-shaped: many query heads over one latent KV head, e.g. 128 heads over
// a 576-dim K / 512-dim V).
//
// With G query heads per KV head the path does G flops per cached byte, so
// at G >= 32 it is bound by math, not HBM; every K/V tile must be reused by
// many heads from on-chip memory.  Work item = (sequence b, KV head g, block
// of 32 query heads, split chunk s); the items of one chunk for all head
// blocks -- and for all sequences, since chunks are ordered split-major --
// run close together, so K/V tiles shared by head blocks and by sequences
// with a common prefix are served from L2.
//
// CTA = 1 producer warp + 8 consumer warps, one CTA per SM.
//  - Producer: one 3-D TMA tensor copy per 32-token tile per tensor; the tile
//    is contiguous in HBM and lands as 64-column segments, each a
//    128-byte-swizzled [32 rows x 128 B] array.  Two stages.
//  - The item's 32 query rows are pre-scaled by scale*log2(e), split into
//    bf16 hi + lo and stored in shared memory with the same swizzle.
//  - Scores: S[32 heads x 32 tokens] = Q . K^T with bf16 mma.sync (fp32
//    accumulate; Q_hi and Q_lo accumulate into the same fragment).  Warp w
//    computes 16 heads x 16 tokens over half of the head dim; the two halves
//    meet in shared memory.
//  - Online softmax: 8 threads per head, 4 tokens each; the running max and
//    sum live in registers of that group; probabilities go to shared memory
//    split into bf16 hi + lo, the per-head rescale factor alongside.
//  - Values: warp w owns output columns [64w, 64w+64) for all 32 heads
//    (fp32 accumulators in registers): O = P_hi . V + P_lo . V.
// Every mbarrier wait is bounded; out-of-range blocks and lengths are
// flagged in the status word, never dereferenced.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kHB = 32;                 // query heads per work item
constexpr int kT = 32;                  // tokens per stage
constexpr int kWarps = 8;               // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kStages = 2;
constexpr int kSegBytes = kT * 128;     // one 64-column segment of a tile (or of Q)
constexpr int kSStride = 36;            // fp32 row stride of the score buffer
constexpr int kPStride = 40;            // bf16 row stride of the probability buffer (80 B)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct MlaShape {
    int dk_segs, dv_segs;               // head dims / 64
    __host__ __device__ int q_bytes() const { return kHB * dk_segs * 128; }     // one of hi/lo
    __host__ __device__ int k_bytes() const { return dk_segs * kSegBytes; }
    __host__ __device__ int v_bytes() const { return dv_segs * kSegBytes; }
    __host__ __device__ int stage_bytes() const { return k_bytes() + v_bytes(); }
};

__host__ __device__ inline size_t mla_smem_bytes(const MlaShape &s) {
    return 1024 + size_t(2) * s.q_bytes() + size_t(kStages) * s.stage_bytes() +
           2 * kHB * kSStride * sizeof(float) + 2 * kHB * kPStride * 2 + 3 * kHB * sizeof(float) +
           2 * kStages * sizeof(uint64_t) + 16;
}

__device__ __forceinline__ int64_t lmin(int64_t x, int64_t y) { return x < y ? x : y; }
__device__ __forceinline__ int64_t lmax(int64_t x, int64_t y) { return x > y ? x : y; }

// Byte offset of (row, 16-byte chunk c) in a segmented, swizzled array of
// 32-row segments.
__device__ __forceinline__ uint32_t seg_addr(int row, int c) {
    return uint32_t(c >> 3) * kSegBytes + uint32_t(row) * 128 + uint32_t(((c & 7) ^ (row & 7)) << 4);
}

struct MlaItem {
    int b, g, hb, s;
    int64_t begin, end;
    int nstages;
};

__device__ __forceinline__ MlaItem mla_item(const DecodeArgs &a, int item, int hblocks,
                                            bool report) {
    MlaItem r;
    const int per_split = a.batch * a.cache.num_kv_heads * hblocks;
    r.s = item / per_split;                 // split-major: a chunk for every row together
    int t = item % per_split;
    r.hb = t % hblocks;
    t /= hblocks;
    r.g = t % a.cache.num_kv_heads;
    r.b = t / a.cache.num_kv_heads;
    int64_t L = a.seq_lens[r.b];
    if (L < 0 || L > int64_t(a.max_blocks) * a.cache.block_size) {
        if (report && r.s == 0 && r.hb == 0) raise_status(a.status, PKV_DEV_SEQ_LEN);
        L = 0;
    }
    const int64_t chunk = 64 * ((L + 64LL * a.num_splits - 1) / (64LL * a.num_splits));
    r.begin = int64_t(r.s) * chunk;
    r.end = lmin(L, r.begin + chunk);
    r.nstages = r.end > r.begin ? int((r.end - r.begin + kT - 1) / kT) : 0;
    return r;
}

__global__ void __launch_bounds__(kThreads, 1)
decode_mla_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a,
                  const MlaShape shp) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_hi = smem;
    uint8_t *q_lo = q_hi + shp.q_bytes();
    uint8_t *stages = q_lo + shp.q_bytes();
    float *sbuf = reinterpret_cast<float *>(stages + size_t(kStages) * shp.stage_bytes());
    uint16_t *pbuf = reinterpret_cast<uint16_t *>(sbuf + 2 * kHB * kSStride);   // hi | lo
    float *abuf = reinterpret_cast<float *>(pbuf + 2 * kHB * kPStride);         // rescale
    float *mbuf = abuf + kHB;                                                   // final m
    float *lbuf = mbuf + kHB;                                                   // final l
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(lbuf + kHB);
    uint64_t *empty_bar = full_bar + kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty_bar + kStages);
    volatile int *cons_abort = abort_flag + 1;   // written by consumers only

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.num_q_heads / a.cache.num_kv_heads;
    const int hblocks = G / kHB;
    const int num_items = a.batch * a.cache.num_kv_heads * hblocks * a.num_splits;
    const int bs = a.cache.block_size;
    const int hkv = a.cache.num_kv_heads;
    const int Dk = shp.dk_segs * 64, Dv = shp.dv_segs * 64;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), kWarps);
        }
        *abort_flag = 0;
        *cons_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait();

    if (warp == kWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        int stage = 0;
        uint32_t phase = 0;
        uint32_t armed = 0, armed_parity = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
            const MlaItem r = mla_item(a, item, hblocks, false);
            const int32_t *table = a.block_tables + int64_t(r.b) * a.max_blocks;
            for (int base = 0; base < r.nstages && ok; base += 32) {
                // Lane i resolves stage base + i; block 0 of this KV head
                // stands in for a stage without a token (never read: all of
                // an item's stages hold a token).
                int32_t y = r.g * bs;
                const int st = base + lane;
                if (st < r.nstages) {
                    const int64_t ts = r.begin + int64_t(st) * kT;
                    const int32_t phys = table[ts / bs];
                    if (phys >= 0 && phys < a.cache.num_blocks)
                        y = (phys * hkv + r.g) * bs + int32_t(ts % bs);
                    else
                        raise_status(a.status, PKV_DEV_BLOCK_ID);
                }
                const int n = min(32, r.nstages - base);
                for (int k = 0; k < n; ++k) {
                    const uint32_t eb = smem_addr(&empty_bar[stage]);
                    const uint32_t fb = smem_addr(&full_bar[stage]);
                    int fail = 0;
                    if (lane == 0) fail = !mbar_wait(eb, phase ^ 1u, a.status) || *abort_flag;
                    if (__shfl_sync(0xffffffffu, fail, 0)) {
                        if (lane == 0) *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    const int32_t yk = __shfl_sync(0xffffffffu, y, k);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(fb, shp.stage_bytes());
                        const uint32_t dst = smem_addr(stages + size_t(stage) * shp.stage_bytes());
                        tma_load_3d(dst, &tmap_k, 0, yk, 0, fb);
                        tma_load_3d(dst + shp.k_bytes(), &tmap_v, 0, yk, 0, fb);
                    }
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        if (lane == 0)
            for (int s = 0; s < kStages; ++s)
                if (armed & (1u << s))
                    mbar_wait(smem_addr(&full_bar[s]), (armed_parity >> s) & 1u, a.status);
        return;
    }

    // -------------------------------------------------------------- consumers
    const int tid = threadIdx.x;                 // 0..255
    const int g8 = lane >> 2, t4 = lane & 3;     // mma fragment coordinates
    // score phase: warp w -> head half, token half, dim half
    const int hh = warp & 1, th = (warp >> 1) & 1, dh = warp >> 2;
    const int ksteps = Dk / 32;                  // per dim half
    // softmax phase: 8 threads per head, 4 tokens each
    const int sm_head = tid >> 3, sm_q = tid & 7;
    // value phase: warp w owns output columns [64w, 64w + 64)
    const bool pv_active = warp < shp.dv_segs;
    const float qscale = a.scale * kLog2e;

    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
        const MlaItem r = mla_item(a, item, hblocks, tid == 0);
        const int head0 = r.g * G + r.hb * kHB;   // first query head of the block

        // ---- load the block's queries: pre-scaled, split hi/lo, swizzled
        {
            // 16-byte loads, eight in flight per thread before any is used
            const float4 *qsrc =
                reinterpret_cast<const float4 *>(a.q + (int64_t(r.b) * a.num_q_heads + head0) * Dk);
            const int n4 = kHB * Dk / 4, nt = kWarps * 32;
            for (int i0 = 0; i0 < n4; i0 += 8 * nt) {
                float4 x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * nt + tid;
                    x[u] = i < n4 ? __ldg(qsrc + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u * nt + tid;
                    if (i >= n4) continue;
                    const int h = (4 * i) / Dk, d = (4 * i) % Dk;
                    const float x0 = x[u].x * qscale, x1 = x[u].y * qscale;
                    const float x2 = x[u].z * qscale, x3 = x[u].w * qscale;
                    const float h0 = __uint_as_float(f32_to_bf16_bits(x0) << 16);
                    const float h1 = __uint_as_float(f32_to_bf16_bits(x1) << 16);
                    const float h2 = __uint_as_float(f32_to_bf16_bits(x2) << 16);
                    const float h3 = __uint_as_float(f32_to_bf16_bits(x3) << 16);
                    // four consecutive dims share one 16-byte chunk
                    const uint32_t off = seg_addr(h, d >> 3) + (d & 7) * 2;
                    *reinterpret_cast<uint2 *>(q_hi + off) =
                        make_uint2(pack_bf16x2(h0, h1), pack_bf16x2(h2, h3));
                    *reinterpret_cast<uint2 *>(q_lo + off) =
                        make_uint2(pack_bf16x2(x0 - h0, x1 - h1), pack_bf16x2(x2 - h2, x3 - h3));
                }
            }
        }
        float acc[2][8][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;
        named_barrier_sync(1, kWarps * 32);       // queries written

        for (int st = 0; st < r.nstages; ++st) {
            // A wait that gives up is published before the barrier below and
            // read after it, so every consumer warp takes the same decision
            // (named barriers do not time out: warps must never diverge here).
            const uint32_t fb = smem_addr(&full_bar[stage]);
            const bool waited = mbar_wait(fb, phase, a.status);
            const bool failed = __any_sync(0xffffffffu, !waited || *abort_flag);
            if (failed && lane == 0) {
                *abort_flag = 1;
                *cons_abort = 1;
            }
            uint8_t *kt = stages + size_t(stage) * shp.stage_bytes();
            uint8_t *vt = kt + shp.k_bytes();
            const int64_t tok0 = r.begin + int64_t(st) * kT;
            const int nvalid = int(lmax(0, lmin(kT, r.end - tok0)));

            if (!failed) {
                // ---- partial scores over this warp's half of the head dim
                float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                const int qrow = hh * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int krow = th * 16 + (lane & 7) + (lane >> 4) * 8;
                const uint32_t qh = smem_addr(q_hi), ql = smem_addr(q_lo), kb = smem_addr(kt);
                for (int kk = 0; kk < ksteps; ++kk) {
                    const int ks = dh * ksteps + kk;                 // 16-dim step
                    const int qc = 2 * ks + (lane >> 4);
                    const int kc = 2 * ks + ((lane >> 3) & 1);
                    uint32_t a0, a1, a2, a3, c0, c1, c2, c3, b0, b1, b2, b3;
                    ldsm_x4(qh + seg_addr(qrow, qc), a0, a1, a2, a3);
                    ldsm_x4(ql + seg_addr(qrow, qc), c0, c1, c2, c3);
                    ldsm_x4(kb + seg_addr(krow, kc), b0, b1, b2, b3);
                    mma_bf16_16816(sacc[0], a0, a1, a2, a3, b0, b1);
                    mma_bf16_16816(sacc[1], a0, a1, a2, a3, b2, b3);
                    mma_bf16_16816(sacc[0], c0, c1, c2, c3, b0, b1);
                    mma_bf16_16816(sacc[1], c0, c1, c2, c3, b2, b3);
                }
                float *sb = sbuf + dh * kHB * kSStride;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int tok = th * 16 + nt * 8 + 2 * t4;
                    const int h = hh * 16 + g8;
                    *reinterpret_cast<float2 *>(sb + h * kSStride + tok) =
                        make_float2(sacc[nt][0], sacc[nt][1]);
                    *reinterpret_cast<float2 *>(sb + (h + 8) * kSStride + tok) =
                        make_float2(sacc[nt][2], sacc[nt][3]);
                }
                // ---- value rows past the end may hold any bits: zero them
                if (nvalid < kT) {
                    const int chunks = (kT - nvalid) * shp.dv_segs * 8;
                    for (int idx = tid; idx < chunks; idx += kWarps * 32) {
                        const int row = nvalid + idx / (shp.dv_segs * 8);
                        const int c = idx % (shp.dv_segs * 8);
                        *reinterpret_cast<uint4 *>(vt + seg_addr(row, c)) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
            }
            named_barrier_sync(1, kWarps * 32);   // scores (and zeroed rows) visible
            ok = *cons_abort == 0;                // the same in every consumer warp

            if (ok) {
                // ---- online softmax, 8 threads per head
                float s[4];
                const int tq = sm_q * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float v = sbuf[sm_head * kSStride + tq + e] +
                                    sbuf[kHB * kSStride + sm_head * kSStride + tq + e];
                    s[e] = (tq + e) < nvalid ? v : -INFINITY;
                }
                float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                const float m_new = fmaxf(m_run, mx);     // finite: the stage has a token
                const float alpha = exp2f(m_run - m_new);
                float psum = 0.f;
                uint16_t ph[4], pl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p = exp2f(s[e] - m_new);
                    psum += p;
                    const uint32_t hb16 = f32_to_bf16_bits(p);
                    ph[e] = uint16_t(hb16);
                    pl[e] = uint16_t(f32_to_bf16_bits(p - __uint_as_float(hb16 << 16)));
                }
                l_run = l_run * alpha + psum;
                m_run = m_new;
                uint16_t *prow_hi = pbuf + sm_head * kPStride + tq;
                uint16_t *prow_lo = pbuf + kHB * kPStride + sm_head * kPStride + tq;
                *reinterpret_cast<uint2 *>(prow_hi) =
                    make_uint2(uint32_t(ph[0]) | (uint32_t(ph[1]) << 16),
                               uint32_t(ph[2]) | (uint32_t(ph[3]) << 16));
                *reinterpret_cast<uint2 *>(prow_lo) =
                    make_uint2(uint32_t(pl[0]) | (uint32_t(pl[1]) << 16),
                               uint32_t(pl[2]) | (uint32_t(pl[3]) << 16));
                if (sm_q == 0) abuf[sm_head] = alpha;
            }
            named_barrier_sync(1, kWarps * 32);   // probabilities visible

            if (ok && pv_active) {
                // ---- O[:, 64w .. 64w+64) = alpha * O + P . V
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const float al0 = abuf[mt * 16 + g8], al1 = abuf[mt * 16 + g8 + 8];
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        acc[mt][nt][0] *= al0; acc[mt][nt][1] *= al0;
                        acc[mt][nt][2] *= al1; acc[mt][nt][3] *= al1;
                    }
                }
                const uint32_t ph_base = smem_addr(pbuf), pl_base = ph_base + kHB * kPStride * 2;
                const uint32_t vb = smem_addr(vt);
#pragma unroll
                for (int kk = 0; kk < kT / 16; ++kk) {
                    uint32_t pa[2][2][4];                      // [hi/lo][m-tile][frag]
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        const int prow = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                        const uint32_t off = prow * kPStride * 2 + (2 * kk + (lane >> 4)) * 16;
                        ldsm_x4(ph_base + off, pa[0][mt][0], pa[0][mt][1], pa[0][mt][2], pa[0][mt][3]);
                        ldsm_x4(pl_base + off, pa[1][mt][0], pa[1][mt][1], pa[1][mt][2], pa[1][mt][3]);
                    }
                    const int vrow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {              // pairs of 8-column n-tiles
                        const int vc = warp * 8 + 2 * j + (lane >> 4);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_trans(vb + seg_addr(vrow, vc), b0, b1, b2, b3);
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                            for (int x = 0; x < 2; ++x) {
                                mma_bf16_16816(acc[mt][2 * j], pa[x][mt][0], pa[x][mt][1],
                                               pa[x][mt][2], pa[x][mt][3], b0, b1);
                                mma_bf16_16816(acc[mt][2 * j + 1], pa[x][mt][0], pa[x][mt][1],
                                               pa[x][mt][2], pa[x][mt][3], b2, b3);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
            if (!ok) break;
        }

        // ---- finalize: per-head max and sum, then each warp writes its columns
        {
            float l = l_run;
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            if (sm_q == 0) {
                mbuf[sm_head] = m_run;
                lbuf[sm_head] = l;
            }
        }
        named_barrier_sync(1, kWarps * 32);
        const int64_t row0 = (int64_t(r.s) * a.batch + r.b) * a.num_q_heads + head0;
        if (pv_active) {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                    const int h = mt * 16 + g8 + 8 * hi;
                    const float l = lbuf[h];
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    float *orow = a.out_part + (row0 + h) * Dv + warp * 64;
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
                        *reinterpret_cast<float2 *>(orow + nt * 8 + 2 * t4) =
                            make_float2(acc[mt][nt][2 * hi] * inv, acc[mt][nt][2 * hi + 1] * inv);
                }
            }
        }
        if (tid < kHB) {
            const float l = lbuf[tid], m = mbuf[tid];
            a.lse_part[row0 + tid] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        }
        named_barrier_sync(1, kWarps * 32);   // buffers free for the next item
    }
}

PFN_cuTensorMapEncodeTiled_v12000 mla_encode_fn() {
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
// (64 columns, rows, dim/64 segments at a 128-byte stride): one box = 32
// rows, all segments -- one contiguous run of HBM for a dense pool --
// landing segment-major.
bool make_seg_map(CUtensorMap *map, const void *pool, int64_t rows, int dim, int stride) {
    auto fn = mla_encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[3] = {64, cuuint64_t(rows), cuuint64_t(dim / 64)};
    cuuint64_t gstride[2] = {cuuint64_t(stride) * 2, 128};
    cuuint32_t box[3] = {64, cuuint32_t(kT), cuuint32_t(dim / 64)};
    cuuint32_t estride[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), gdim, gstride,
              box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mla_kernel_supports(const pkv_cache_desc &c, int32_t num_q_heads) {
    const int G = num_q_heads / c.num_kv_heads;
    const bool pow2_bs = c.block_size >= kT && c.block_size <= 256 &&
                         (c.block_size & (c.block_size - 1)) == 0;
    const int64_t rows = int64_t(c.num_blocks) * c.num_kv_heads * c.block_size;
    if (G % kHB != 0 || !pow2_bs || rows >= (int64_t(1) << 31) - 1) return false;
    if (c.head_dim_k % 64 != 0 || c.head_dim_v % 64 != 0) return false;
    if (c.head_dim_v > 64 * kWarps || c.head_dim_k < 64) return false;
    const MlaShape s{c.head_dim_k / 64, c.head_dim_v / 64};
    return mla_smem_bytes(s) <= 232448;
}

int32_t mla_work_units(const pkv_cache_desc &c, int32_t batch, int32_t num_q_heads) {
    return batch * num_q_heads / kHB;
}

int launch_decode_mla(const DecodeArgs &a) {
    const MlaShape shp{a.cache.head_dim_k / 64, a.cache.head_dim_v / 64};
    const int64_t rows = int64_t(a.cache.num_blocks) * a.cache.num_kv_heads * a.cache.block_size;
    CUtensorMap tk, tv;
    if (!make_seg_map(&tk, a.k_pool, rows, a.cache.head_dim_k, a.cache.head_dim_k) ||
        !make_seg_map(&tv, a.v_pool, rows, a.cache.head_dim_v, a.v_stride))
        return PKV_ERR_CUDA;
    const size_t smem = mla_smem_bytes(shp);
    static thread_local int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        if (cudaFuncSetAttribute(decode_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 232448) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_dev = dev;
    }
    const int G = a.num_q_heads / a.cache.num_kv_heads;
    const int64_t items = int64_t(a.batch) * a.cache.num_kv_heads * (G / kHB) * a.num_splits;
    const int grid = int(std::min<int64_t>(items, sm_count()));
    if (grid <= 0) return PKV_OK;
    return launch_pdl(decode_mla_kernel, dim3(grid), dim3(kThreads), smem, a.stream, tk, tv, a,
                      shp);
}

}  // namespace pkv
