// merge.cu -- standalone log-sum-exp merge of two attention partials (the online-softmax merge
// equation of the Context-Parallel page, section 先弄清楚): l = log(e^l1 + e^l2),
// o = e^(l1 - l) o1 + e^(l2 - l) o2, evaluated as l = max + log1p(e^-|l1 - l2|) in fp32.
// HBM-bound: every row reads two lse values and two hd-vectors and writes one of each.
#include <math.h>

#include "usp_internal.cuh"
#include "usp_device.cuh"

namespace usp {
namespace {

// 16-byte unit <-> 8 bf16 or 4 fp32 values
template <typename T> struct Unit;
template <> struct Unit<float> {
    static constexpr int N = 4;
    __device__ static void load(const void *p, float *x) {
        float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    __device__ static void store(void *p, const float *x) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};
template <> struct Unit<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const void *p, float *x) {
        uint4 v = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = bf16x2_to_float2(w[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    __device__ static void store(void *p, const float *x) {
        uint4 v;
        v.x = float2_to_bf16x2(x[0], x[1]);
        v.y = float2_to_bf16x2(x[2], x[3]);
        v.z = float2_to_bf16x2(x[4], x[5]);
        v.w = float2_to_bf16x2(x[6], x[7]);
        *reinterpret_cast<uint4 *>(p) = v;
    }
};

template <typename T>
__global__ void __launch_bounds__(256) lse_merge_kernel(T *o_acc, float *lse_acc, const T *o_new,
                                                        const float *lse_new, uint32_t rows, uint32_t upr,
                                                        uint32_t rows_per_warp) {
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    // rows_per_warp > 0: each warp handles rows_per_warp whole rows at a time (upr divides 32);
    // otherwise one row per warp with the lanes striding over its units.
    const uint32_t lanes_per_row = rows_per_warp ? upr : 32;
    const uint32_t rsub = rows_per_warp ? lane / upr : 0;
    const uint32_t col0 = rows_per_warp ? lane % upr : lane;
    const uint32_t step_rows = rows_per_warp ? rows_per_warp : 1;
    for (uint32_t r0 = warp * step_rows; r0 < rows; r0 += nwarps * step_rows) {
        const uint32_t row = r0 + rsub;
        const bool active = row < rows && (rows_per_warp == 0 || rsub < rows_per_warp);
        float w1 = 0.f, w2 = 0.f, l = -INFINITY;
        if (active) merge_weights(lse_acc[row], lse_new[row], w1, w2, l);
        __syncwarp();  // every lane has read lse_acc[row] before it is rewritten below
        if (active) {
            for (uint32_t col = col0; col < upr; col += lanes_per_row) {
                const size_t off = ((size_t)row * upr + col) * Unit<T>::N;
                float a[Unit<T>::N], b[Unit<T>::N];
                Unit<T>::load(o_acc + off, a);
                Unit<T>::load(o_new + off, b);
#pragma unroll
                for (int e = 0; e < Unit<T>::N; ++e) a[e] = w1 * a[e] + w2 * b[e];
                Unit<T>::store(o_acc + off, a);
            }
            if (col0 == 0) lse_acc[row] = l;
        }
    }
}

}  // namespace

int launch_lse_merge(void *o_acc, float *lse_acc, const void *o_new, const float *lse_new, int64_t rows,
                     int hd, int dtype, cudaStream_t s) {
    const DeviceInfo *di = device_info();
    if (!di) return USP_ERR_CUDA;
    const uint32_t upr = (uint32_t)((int64_t)hd * elem_size(dtype) / 16);
    const uint32_t rpw = (upr <= 32 && 32 % upr == 0) ? 32 / upr : 0;
    const int64_t warps_needed = rpw ? (rows + rpw - 1) / rpw : rows;
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = (int64_t)di->sm_count * 16;
    if (blocks > cap) blocks = cap;
    if (dtype == USP_F32)
        lse_merge_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(
            static_cast<float *>(o_acc), lse_acc, static_cast<const float *>(o_new), lse_new, (uint32_t)rows,
            upr, rpw);
    else
        lse_merge_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
            static_cast<__nv_bfloat16 *>(o_acc), lse_acc, static_cast<const __nv_bfloat16 *>(o_new), lse_new,
            (uint32_t)rows, upr, rpw);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace usp
