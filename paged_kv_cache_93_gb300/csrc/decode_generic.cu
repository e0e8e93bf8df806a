// decode_generic.cu -- the generic CUDA-core decode-attention kernel and the
// LSE merge kernel.
//
// Generic kernel: one warp per (sequence, query head, split).  Lanes split the
// head dimension into 16-byte bf16 vectors; each token's score is a warp
// reduction, and the online softmax (running max m, running sum l, rescaled
// accumulator) runs in base 2 with the query pre-multiplied by scale*log2(e).
// A warp takes kU tokens per step -- their K rows loaded together, then their
// V rows -- so kU row loads are in flight instead of one.
// It handles any head dims (multiples of 8 up to 1024), any query group and
// any block size; the TMA + tensor-core kernel covers the common GQA shapes.
// With E4 set the pools hold E4M3 codes (8 bytes per 8 elements, decoded
// exactly through fp16); the key scale folds into the query and the value
// scale into the final 1/l.
// The LSE merge kernel lives here too.
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kGenericWarps = 4;
constexpr int kU = 4;                   // tokens per step of a warp

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    f[0] = bf16_lo_to_f32(u.x); f[1] = bf16_hi_to_f32(u.x);
    f[2] = bf16_lo_to_f32(u.y); f[3] = bf16_hi_to_f32(u.y);
    f[4] = bf16_lo_to_f32(u.z); f[5] = bf16_hi_to_f32(u.z);
    f[6] = bf16_lo_to_f32(u.w); f[7] = bf16_hi_to_f32(u.w);
}

// 8 E4M3 codes -> their values.
__device__ __forceinline__ void unpack8_e4m3(const uint2 &u, float (&f)[8]) {
    const float2 a = e4m3x2_to_f32(u.x & 0xffffu), b = e4m3x2_to_f32(u.x >> 16);
    const float2 c = e4m3x2_to_f32(u.y & 0xffffu), d = e4m3x2_to_f32(u.y >> 16);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// Elements 8v .. 8v+7 of row `row` of a pool whose rows hold `n8` groups of 8,
// as stored (16 bytes of bf16 or 8 bytes of E4M3 codes), and their values.
template <bool E4>
using Raw8 = typename std::conditional<E4, uint2, uint4>::type;
template <bool E4>
__device__ __forceinline__ Raw8<E4> load_raw8(const void *pool, int64_t row, int n8, int v) {
    return static_cast<const Raw8<E4> *>(pool)[row * n8 + v];
}
__device__ __forceinline__ void unpack8_any(const uint4 &u, float (&f)[8]) { unpack8(u, f); }
__device__ __forceinline__ void unpack8_any(const uint2 &u, float (&f)[8]) { unpack8_e4m3(u, f); }

// KC / VC: 8-element groups per lane for K and V (ceil(dim / 8 / 32)).
template <int KC, int VC, bool E4>
__global__ void __launch_bounds__(kGenericWarps * 32)
decode_generic_kernel(DecodeArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int h = blockIdx.y * kGenericWarps + (threadIdx.x >> 5);
    const int b = blockIdx.z;
    const int split = blockIdx.x;
    if (h >= a.num_q_heads) return;
    const pkv_cache_desc &c = a.cache;
    const int group = a.num_q_heads / c.num_kv_heads;
    const int g = h / group;
    const int nk = c.head_dim_k / 8, nv = c.head_dim_v / 8;

    int64_t L = a.seq_lens[b];
    if (L < 0 || L > int64_t(a.max_blocks) * c.block_size) {
        if (lane == 0 && split == 0 && (h % group) == 0) raise_status(a.status, PKV_DEV_SEQ_LEN);
        L = 0;
    }
    const int64_t chunk = 64 * ((L + 64LL * a.num_splits - 1) / (64LL * a.num_splits));
    const int64_t begin = int64_t(split) * chunk;
    const int64_t end = L < begin + chunk ? L : begin + chunk;

    // q, pre-scaled so that scores come out in base-2 log units.
    float qv[KC][8];
    const float qscale = a.scale * kLog2e * (E4 ? a.k_scale[g] : 1.f);
    const float *qrow = a.q + (int64_t(b) * a.num_q_heads + h) * c.head_dim_k;
#pragma unroll
    for (int i = 0; i < KC; ++i) {
        const int v = lane + 32 * i;
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[i][e] = v < nk ? qrow[v * 8 + e] * qscale : 0.f;
    }
    float acc[VC][8];
#pragma unroll
    for (int i = 0; i < VC; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
    float m = -INFINITY, l = 0.f;

    const int32_t *table = a.block_tables + int64_t(b) * a.max_blocks;
    const int vs = a.v_stride / 8;          // 8-element groups from one V row to the next
    for (int64_t j0 = begin; j0 < end; j0 += kU) {
        // tokens j0 .. j0 + kU - 1; those at or past `end` score -inf.  A
        // block id out of range is flagged and its token reads as zeros.
        int64_t row[kU];
        bool live[kU], ok[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t j = j0 + u;
            live[u] = j < end;
            const int32_t phys = live[u] ? table[j / c.block_size] : 0;
            ok[u] = live[u] && phys >= 0 && phys < c.num_blocks;
            if (live[u] && !ok[u] && lane == 0 && (h % group) == 0)
                raise_status(a.status, PKV_DEV_BLOCK_ID);
            row[u] = (int64_t(ok[u] ? phys : 0) * c.num_kv_heads + g) * c.block_size +
                     j % c.block_size;
        }
        Raw8<E4> kr[kU][KC];
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
            for (int i = 0; i < KC; ++i) {
                const int v = lane + 32 * i;
                kr[u][i] = v < nk && ok[u] ? load_raw8<E4>(a.k_pool, row[u], nk, v) : Raw8<E4>{};
            }
        float sc[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < KC; ++i) {
                float kf[8];
                unpack8_any(kr[u][i], kf);
#pragma unroll
                for (int e = 0; e < 8; ++e) part = fmaf(qv[i][e], kf[e], part);
            }
            sc[u] = part;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) sc[u] = live[u] ? warp_sum(sc[u]) : -INFINITY;
        float m_new = m;
#pragma unroll
        for (int u = 0; u < kU; ++u) m_new = fmaxf(m_new, sc[u]);
        const float corr = exp2f(m - m_new);
        float p[kU], psum = 0.f;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            p[u] = exp2f(sc[u] - m_new);
            psum += p[u];
        }
        l = l * corr + psum;
        m = m_new;
        Raw8<E4> vr[kU][VC];
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
            for (int i = 0; i < VC; ++i) {
                const int v = lane + 32 * i;
                vr[u][i] = v < nv && ok[u] ? load_raw8<E4>(a.v_pool, row[u], vs, v) : Raw8<E4>{};
            }
#pragma unroll
        for (int i = 0; i < VC; ++i) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] *= corr;
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                float vf[8];
                unpack8_any(vr[u][i], vf);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(p[u], vf[e], acc[i][e]);
            }
        }
    }

    const int64_t orow = (int64_t(split) * a.batch + b) * a.num_q_heads + h;
    const float inv = l > 0.f ? (E4 ? a.v_scale[g] : 1.f) / l : 0.f;
    float *o = a.out_part + orow * c.head_dim_v;
#pragma unroll
    for (int i = 0; i < VC; ++i) {
        const int v = lane + 32 * i;
        if (v < nv) {
            float4 lo = make_float4(acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv);
            float4 hi = make_float4(acc[i][4] * inv, acc[i][5] * inv, acc[i][6] * inv, acc[i][7] * inv);
            reinterpret_cast<float4 *>(o)[2 * v] = lo;
            reinterpret_cast<float4 *>(o)[2 * v + 1] = hi;
        }
    }
    if (lane == 0) a.lse_part[orow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// Dv/4 threads per row, one float4 of the output each.  The partials are
// taken 16 at a time: all 16 LSEs and output float4s of a chunk are loaded
// at once (independent loads, one memory round trip), then folded into a
// running (max, weight sum, weighted sum) that is rescaled whenever the max
// grows -- the same exact merge, in chunks.
__global__ void lse_merge_kernel(int32_t num_parts, const float *__restrict__ out_part,
                                 const float *__restrict__ lse_part, int64_t rows,
                                 int32_t head_dim_v, float *__restrict__ out,
                                 float *__restrict__ lse) {
    pdl_wait();
    pdl_launch_dependents();
    const int tpr = head_dim_v / 4;
    const int64_t r = blockIdx.x * int64_t(blockDim.x / tpr) + threadIdx.x / tpr;
    const int c = threadIdx.x % tpr;
    if (r >= rows) return;
    const float4 *op = reinterpret_cast<const float4 *>(out_part + r * head_dim_v) + c;
    const int64_t pstride = rows * tpr;   // float4s between consecutive partials
    float M = -INFINITY, W = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool nan_part = false;     // a partial reported as NaN (abandoned): the row is NaN
    for (int p0 = 0; p0 < num_parts; p0 += 16) {
        float l[16];
        float4 x[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const bool in = p0 + u < num_parts;
            l[u] = in ? lse_part[int64_t(p0 + u) * rows + r] : -INFINITY;
            x[u] = in ? op[int64_t(p0 + u) * pstride] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mc = M;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            nan_part |= l[u] != l[u];
            mc = fmaxf(mc, l[u]);
        }
        if (mc == -INFINITY) continue;               // every partial so far is empty
        const float rescale = expf(M - mc);          // 0 when M = -inf
        W *= rescale;
        acc = make_float4(acc.x * rescale, acc.y * rescale, acc.z * rescale, acc.w * rescale);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const float w = expf(l[u] - mc);
            // An empty partial has w = 0 and out = 0; skip it so stray values
            // in an empty partial's output cannot reach the sum.
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

template <int KC, int VC, bool E4>
int launch_generic(const DecodeArgs &a) {
    dim3 grid(a.num_splits, (a.num_q_heads + kGenericWarps - 1) / kGenericWarps, a.batch);
    return launch_pdl(decode_generic_kernel<KC, VC, E4>, grid, dim3(kGenericWarps * 32), 0,
                      a.stream, a);
}

template <bool E4>
int launch_generic_dims(const DecodeArgs &a) {
    const int kc = (a.cache.head_dim_k / 8 + 31) / 32;
    const int vc = (a.cache.head_dim_v / 8 + 31) / 32;
    if (kc <= 1 && vc <= 1) return launch_generic<1, 1, E4>(a);
    if (kc <= 2 && vc <= 2) return launch_generic<2, 2, E4>(a);
    if (kc <= 3 && vc <= 2) return launch_generic<3, 2, E4>(a);
    return launch_generic<4, 4, E4>(a);
}

}  // namespace

int launch_decode_generic(const DecodeArgs &a) { return launch_generic_dims<false>(a); }

int launch_decode_generic_e4m3(const DecodeArgs &a) { return launch_generic_dims<true>(a); }

int launch_lse_merge(int32_t num_parts, const float *out_part, const float *lse_part,
                     int64_t rows, int32_t head_dim_v, float *out, float *lse,
                     cudaStream_t stream) {
    // Two rows per CTA for Dv = 128 (64 threads): enough CTAs to spread even
    // a few hundred rows over the SMs.
    const int tpr = head_dim_v / 4;
    const int rows_per_cta = tpr >= 64 ? 1 : 64 / tpr;
    const int64_t blocks = (rows + rows_per_cta - 1) / rows_per_cta;
    return launch_pdl(lse_merge_kernel, dim3(static_cast<unsigned>(blocks)),
                      dim3(rows_per_cta * tpr), 0, stream, num_parts, out_part, lse_part, rows,
                      head_dim_v, out, lse);
}

}  // namespace pkv
