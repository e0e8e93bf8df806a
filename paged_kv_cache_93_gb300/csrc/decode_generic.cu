// decode_generic.cu -- the generic CUDA-core decode-attention kernel and the
// LSE merge kernel.
//
// Generic kernel: one warp per (sequence, query head, split).  Lanes split the
// head dimension into 16-byte bf16 vectors; each token's score is a warp
// reduction, and the online softmax (running max m, running sum l, rescaled
// accumulator) runs in base 2 with the query pre-multiplied by scale*log2(e).
// It handles any head dims (multiples of 8 up to 1024), any query group and
// any block size; the TMA + tensor-core kernel covers the common GQA shapes.
#include <cuda_runtime.h>

#include <algorithm>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kGenericWarps = 4;

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

// KC / VC: 16-byte vectors per lane for K and V (ceil(dim / 8 / 32)).
template <int KC, int VC>
__global__ void __launch_bounds__(kGenericWarps * 32)
decode_generic_kernel(DecodeArgs a) {
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
    const float qscale = a.scale * kLog2e;
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
    const uint4 *kp = static_cast<const uint4 *>(a.k_pool);
    const uint4 *vp = static_cast<const uint4 *>(a.v_pool);
    for (int64_t j = begin; j < end; ++j) {
        const int32_t phys = table[j / c.block_size];
        const bool ok = phys >= 0 && phys < c.num_blocks;
        if (!ok && lane == 0 && (h % group) == 0) raise_status(a.status, PKV_DEV_BLOCK_ID);
        const int64_t row = (int64_t(ok ? phys : 0) * c.num_kv_heads + g) * c.block_size +
                            j % c.block_size;
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < KC; ++i) {
            const int v = lane + 32 * i;
            if (v < nk && ok) {
                float kf[8];
                unpack8(kp[row * nk + v], kf);
#pragma unroll
                for (int e = 0; e < 8; ++e) part = fmaf(qv[i][e], kf[e], part);
            }
        }
        const float s = warp_sum(part);
        const float m_new = fmaxf(m, s);
        const float corr = exp2f(m - m_new);
        const float p = exp2f(s - m_new);
        l = l * corr + p;
        m = m_new;
#pragma unroll
        for (int i = 0; i < VC; ++i) {
            const int v = lane + 32 * i;
            float vf[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (v < nv && ok) unpack8(vp[row * nv + v], vf);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(p, vf[e], acc[i][e] * corr);
        }
    }

    const int64_t orow = (int64_t(split) * a.batch + b) * a.num_q_heads + h;
    const float inv = l > 0.f ? 1.f / l : 0.f;
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

// One warp per row: pass 1 finds the largest partial LSE, pass 2 sums the
// weights e^(lse_p - M) and the weighted partial outputs.
__global__ void lse_merge_kernel(int32_t num_parts, const float *__restrict__ out_part,
                                 const float *__restrict__ lse_part, int64_t rows,
                                 int32_t head_dim_v, float *__restrict__ out,
                                 float *__restrict__ lse) {
    const int lane = threadIdx.x & 31;
    const int64_t r = blockIdx.x * int64_t(blockDim.x / 32) + (threadIdx.x >> 5);
    if (r >= rows) return;
    float M = -INFINITY;
    for (int p = lane; p < num_parts; p += 32) M = fmaxf(M, lse_part[int64_t(p) * rows + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const int nv4 = head_dim_v / 4;
    float4 *orow = reinterpret_cast<float4 *>(out + r * head_dim_v);
    if (M == -INFINITY) {
        for (int v = lane; v < nv4; v += 32) orow[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane == 0) lse[r] = -INFINITY;
        return;
    }
    float W = 0.f;
    for (int p = 0; p < num_parts; ++p) W += __expf(lse_part[int64_t(p) * rows + r] - M);
    const float inv = 1.f / W;
    for (int v = lane; v < nv4; v += 32) {
        float4 accv = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < num_parts; ++p) {
            const float w = __expf(lse_part[int64_t(p) * rows + r] - M);
            if (w == 0.f) continue;
            const float4 x =
                reinterpret_cast<const float4 *>(out_part + (int64_t(p) * rows + r) * head_dim_v)[v];
            accv.x = fmaf(w, x.x, accv.x); accv.y = fmaf(w, x.y, accv.y);
            accv.z = fmaf(w, x.z, accv.z); accv.w = fmaf(w, x.w, accv.w);
        }
        orow[v] = make_float4(accv.x * inv, accv.y * inv, accv.z * inv, accv.w * inv);
    }
    if (lane == 0) lse[r] = M + logf(W);
}

template <int KC, int VC>
int launch_generic(const DecodeArgs &a) {
    dim3 grid(a.num_splits, (a.num_q_heads + kGenericWarps - 1) / kGenericWarps, a.batch);
    decode_generic_kernel<KC, VC><<<grid, kGenericWarps * 32, 0, a.stream>>>(a);
    return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_decode_generic(const DecodeArgs &a) {
    const int kc = (a.cache.head_dim_k / 8 + 31) / 32;
    const int vc = (a.cache.head_dim_v / 8 + 31) / 32;
    if (kc <= 1 && vc <= 1) return launch_generic<1, 1>(a);
    if (kc <= 2 && vc <= 2) return launch_generic<2, 2>(a);
    if (kc <= 3 && vc <= 2) return launch_generic<3, 2>(a);
    return launch_generic<4, 4>(a);
}

int launch_lse_merge(int32_t num_parts, const float *out_part, const float *lse_part,
                     int64_t rows, int32_t head_dim_v, float *out, float *lse,
                     cudaStream_t stream) {
    const int warps = 8;
    const int64_t blocks = (rows + warps - 1) / warps;
    lse_merge_kernel<<<static_cast<unsigned>(blocks), warps * 32, 0, stream>>>(
        num_parts, out_part, lse_part, rows, head_dim_v, out, lse);
    return cuda_status(cudaGetLastError());
}

}  // namespace pkv
