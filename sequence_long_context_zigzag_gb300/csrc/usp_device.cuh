// usp_device.cuh -- small device helpers shared by the library's kernels (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

namespace usp {

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&w);
    return __bfloat1622float2(h);
}

// round to nearest even; x goes to the low half
__device__ __forceinline__ uint32_t float2_to_bf16x2(float x, float y) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Weights of the log-sum-exp merge of two partials with log-normalisers l1, l2:
// l = log(e^l1 + e^l2) = max(l1, l2) + log1p(e^-|l1 - l2|), w_i = e^(l_i - l).
// -inf marks an empty partial (weight 0); two empty partials give l = -inf, w1 = w2 = 0.
__device__ __forceinline__ void merge_weights(float l1, float l2, float &w1, float &w2, float &l) {
    const bool e1 = (l1 == -INFINITY), e2 = (l2 == -INFINITY);
    if (e1 && e2) {
        w1 = 0.f;
        w2 = 0.f;
        l = -INFINITY;
        return;
    }
    const float m = fmaxf(l1, l2);
    l = m + log1pf(expf(-fabsf(l1 - l2)));
    w1 = e1 ? 0.f : expf(l1 - l);
    w2 = e2 ? 0.f : expf(l2 - l);
}

}  // namespace usp
