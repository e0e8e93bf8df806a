// pkv_math.cuh -- arithmetic helpers of the tcgen05 decode kernels' softmax.
#pragma once

namespace pkv {

// 2^x by the SFU's approximate base-2 exponential (PTX ex2.approx.ftz.f32:
// about 2 ulp; -inf gives +0, subnormal results flush to 0).  For softmax
// weights, whose sums and ratios tolerate far more than that.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace pkv
