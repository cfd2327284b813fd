// usp_internal.cuh -- helpers shared by the library's CUDA translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "usp.h"

namespace usp {

// Division of a 32-bit unsigned numerator n < 2^31 by a runtime divisor d >= 1 with one multiply-high
// and one shift (Granlund & Montgomery, "Division by invariant integers using multiplication", 1994):
// with l = ceil(log2 d) and m = ceil(2^(31+l) / d), floor(n m / 2^(31+l)) == floor(n / d). The error
// term n (m d - 2^(31+l)) / (d 2^(31+l)) is below 2^-l <= 1/d, so it never crosses an integer.
// m fits in 32 bits because d > 2^(l-1).
struct FastDiv {
    uint32_t d;
    uint32_t m;
    uint32_t s;  // shift applied to the high word: l - 1
    FastDiv() : d(1), m(0), s(0) {}
    explicit FastDiv(uint32_t div) : d(div) {
        if (div <= 1) { d = 1; m = 0; s = 0; return; }
        uint32_t l = 0;
        while ((1ull << l) < div) ++l;
        m = (uint32_t)(((1ull << (31 + l)) + div - 1) / div);
        s = l - 1;
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        return d == 1 ? n : (__umulhi(n, m) >> s);
    }
    __device__ __forceinline__ void divmod(uint32_t n, uint32_t &q, uint32_t &r) const {
        q = div(n);
        r = n - q * d;
    }
};

// zigzag position of ring-local row p on ring rank r (chunk length c, ring degree rd):
// rank r keeps global chunks r and 2 rd - 1 - r, in that order.
__host__ __device__ __forceinline__ int64_t zig_pos(int64_t r, int64_t p, int64_t c, int64_t rd) {
    return p < c ? r * c + p : (2 * rd - 1 - r) * c + (p - c);
}

// global position of ring-local row p on ring rank r under a split (usp_split); Lr = 2 c rows per rank
__host__ __device__ __forceinline__ int64_t split_pos(int split, int64_t r, int64_t p, int64_t c, int64_t rd) {
    if (split == USP_SPLIT_BASIC) return r * 2 * c + p;
    if (split == USP_SPLIT_STRIPE) return p * rd + r;
    return zig_pos(r, p, c, rd);
}

// number of ring-local rows of rank s whose global position is <= qpos; every split's position map
// is increasing in the row, so those rows are a prefix
__host__ __device__ __forceinline__ int64_t split_visible(int split, int64_t qpos, int64_t s, int64_t c,
                                                          int64_t rd) {
    const int64_t Lr = 2 * c;
    if (split == USP_SPLIT_BASIC) {
        const int64_t v = qpos - s * Lr + 1;
        return v < 0 ? 0 : (v > Lr ? Lr : v);
    }
    if (split == USP_SPLIT_STRIPE) {
        if (qpos < s) return 0;
        const int64_t v = (qpos - s) / rd + 1;
        return v > Lr ? Lr : v;
    }
    int64_t c0 = qpos - s * c + 1;
    c0 = c0 < 0 ? 0 : (c0 > c ? c : c0);
    int64_t c1 = qpos - (2 * rd - 1 - s) * c + 1;
    c1 = c1 < 0 ? 0 : (c1 > c ? c : c1);
    return c0 + c1;
}

// Packed samples: the first and one-past-last global position [a, e) of the sample holding position
// g, by binary search in the cumulative lengths cu[0..nseq] (read-only, in bounds for any values);
// the result is clamped to a <= g < e <= L, so malformed lengths give odd masks but never a fault.
__device__ __forceinline__ void sample_bounds(const int32_t *cu, uint32_t nseq, uint32_t g, uint32_t L, uint32_t &a,
                                              uint32_t &e) {
    uint32_t lo = 0, hi = nseq;  // the sample index lies in [lo, hi)
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= (int32_t)g) lo = mid;
        else hi = mid;
    }
    const int32_t a0 = __ldg(cu + lo), e0 = __ldg(cu + lo + 1);
    a = (a0 < 0 || (uint32_t)a0 > g) ? (a0 < 0 ? 0u : g) : (uint32_t)a0;
    e = (e0 <= (int32_t)g) ? g + 1 : ((uint32_t)e0 > L ? L : (uint32_t)e0);
}

// per-device cached properties and the device status word address
struct DeviceInfo {
    int sm_count;
    int *status;  // device address of this library's status word on that device
};
// returns nullptr on a CUDA failure
const DeviceInfo *device_info();

inline int elem_size(int dtype) { return dtype == USP_F32 ? 4 : (dtype == USP_BF16 ? 2 : 0); }

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Heads per Ulysses rank after the forward all-to-all of a tensor with H heads: H / ud when ud
// divides H; 1 when H divides ud (K/V of GQA/MQA with fewer heads than Ulysses ranks: every rank
// receives a replica of the one head its query heads read, head u' / (ud / H)); 0 otherwise.
inline int heads_per_rank(int64_t H, int64_t ud) {
    if (H <= 0 || ud <= 0) return 0;
    if (H % ud == 0) return (int)(H / ud);
    return ud % H == 0 ? 1 : 0;
}

// kernel launchers implemented in separate translation units; return USP_* codes
enum PermMode {
    PERM_EXTRACT = 0,      // natural -> local (a1)
    PERM_EXTRACT_INV = 1,  // local -> natural (a7)
    PERM_A2A_FWD = 2,      // local -> head-sharded (a2)
    PERM_A2A_INV = 3,      // head-sharded -> local (a5)
    PERM_FUSED_FWD = 4,    // natural -> head-sharded (a2 after a1)
    PERM_FUSED_INV = 5     // head-sharded -> natural (a7 after a5)
};

constexpr int kMaxPermJobs = 4;

// One tensor moved by a permute launch; every tensor of a launch shares the mode and the grid, and
// may differ in its head window and its row (e.g. out rows of hd elements and lse rows of one fp32).
struct PermJob {
    const char *src;
    char *dst;
    int32_t H, H_total, h0;
    int64_t row_bytes;  // bytes of one (token, head) row: a multiple of 4
    int32_t dtype;      // element type (the replica sum of an inverse all-to-all adds values)
};

struct PermArgs {
    int mode;
    int split;
    int njobs;
    PermJob job[kMaxPermJobs];
    int64_t bs, L;
    int32_t rd, ud;
    int32_t r_fixed, u_fixed;  // >= 0 when only one virtual rank takes part (extract only)
    int32_t max_blocks;        // > 0: at most this many thread blocks (grid-stride), else the default
};
int launch_permute(const PermArgs &a, cudaStream_t s);

int launch_lse_merge(void *o_acc, float *lse_acc, const void *o_new, const float *lse_new, int64_t rows,
                     int hd, int dtype, cudaStream_t s);

struct AttnArgs {
    const void *q, *k, *v;
    void *out;
    float *lse;
    int64_t bs, L;
    int32_t hq, hkv, hd, rd, ud, dtype, causal, mode, step, split, ring_rank_only;
    float scale;
    const int32_t *cu;  // packed samples' cumulative lengths (nseq + 1 entries), or nullptr
    int32_t nseq;       // > 1 when packed
    int32_t max_ctas;   // > 0: the persistent tensor-core kernel runs at most this many CTAs
};
int launch_attn_simt(const AttnArgs &a, cudaStream_t s);
int launch_attn_tc(const AttnArgs &a, cudaStream_t s);

// usp_extract_a2a and usp_attn_fwd with a cap on the SMs they take (0: no cap), for pipelines that
// keep a few SMs free for another stream's kernels
int extract_a2a_capped(int n, const void *const *src, void *const *dst, const usp_dims *d, int inverse,
                       int max_blocks, usp_stream_t stream);
int attn_fwd_capped(const void *q, const void *k, const void *v, void *out, float *lse, const usp_attn_desc &d,
                    int max_ctas, usp_stream_t stream);

// backward: the forward's arguments plus dout, delta and the three gradients
struct BwdArgs {
    AttnArgs f;
    const void *dout;
    const float *delta;
    void *dq, *dk, *dv;
};
int launch_attn_bwd_simt(const BwdArgs &a, cudaStream_t s);
int launch_attn_bwd_tc(const BwdArgs &a, cudaStream_t s);
int launch_row_dot(const void *x, const void *y, float *out, int64_t rows, int hd, int dtype, cudaStream_t s);

}  // namespace usp
