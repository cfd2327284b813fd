// tc_common.cuh -- pieces shared by the tensor-core attention kernels (forward and backward): the
// 32-bit position maps of the sequence splits and the TMA tensor-map encoding (not part of the ABI).
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "usp_internal.cuh"

namespace usp {

// global position of ring-local row p on ring rank r (chunk length c = Lr / 2) under the split:
// zigzag keeps chunks r and 2 rd - 1 - r, basic the contiguous block r, stripe every rd-th token
__device__ __forceinline__ uint32_t pos32(int split, uint32_t r, uint32_t p, uint32_t c, uint32_t rd) {
    if (split == USP_SPLIT_BASIC) return r * 2 * c + p;
    if (split == USP_SPLIT_STRIPE) return p * rd + r;
    return p < c ? r * c + p : (2 * rd - 1 - r) * c + (p - c);
}

// number of ring-local rows of rank s whose global position is <= qpos (a prefix: every split's
// position map is increasing in the row)
__device__ __forceinline__ uint32_t vis32(int split, uint32_t qpos, uint32_t s, uint32_t c, uint32_t rd) {
    if (split == USP_SPLIT_BASIC) {
        const uint32_t a0 = s * 2 * c;
        return qpos < a0 ? 0u : min(qpos - a0 + 1, 2 * c);
    }
    if (split == USP_SPLIT_STRIPE) return qpos < s ? 0u : min((qpos - s) / rd + 1, 2 * c);
    const uint32_t a0 = s * c, a1 = (2 * rd - 1 - s) * c;
    const uint32_t c0 = qpos < a0 ? 0u : min(qpos - a0 + 1, c);
    const uint32_t c1 = qpos < a1 ? 0u : min(qpos - a1 + 1, c);
    return c0 + c1;
}

// number of ring-local rows of rank s whose global position is < kpos (0 when kpos is 0)
__device__ __forceinline__ uint32_t before32(int split, uint32_t kpos, uint32_t s, uint32_t c, uint32_t rd) {
    return kpos == 0 ? 0u : vis32(split, kpos - 1, s, c, rd);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the driver's cuTensorMapEncodeTiled, looked up once through the runtime (no link-time dependency
// on the driver library)
inline EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(f);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// 2-D view (rows x hd) of a bf16 tensor, box_rows-row x 64-column boxes, 128-byte swizzle, zero fill
inline bool make_tmap(CUtensorMap *m, const void *base, uint64_t rows, int hd, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace usp
