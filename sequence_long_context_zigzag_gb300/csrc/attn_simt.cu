// attn_simt.cu -- ring attention forward on the CUDA cores (fp32 arithmetic), one warp per query row.
//
// This is the path for fp32 inputs (and the numerics cross-check for the tensor-core kernel): each
// warp owns one query row of one virtual rank, walks the ring in the order of the Context-Parallel
// page's Fig. 1 (step t: KV block of ring rank (r - t) mod rd), and folds every key into a running
// online softmax (the LSE merge of that page's section 先弄清楚 applied key by key). Because every
// split's position map is increasing within a rank, the keys a causal row sees in a rank's block
// are a prefix of that block, so masking is a loop bound.
#include <math.h>

#include "usp_device.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

struct AttnK {
    const void *q, *k, *v;
    void *out;
    float *lse;
    uint32_t nrows, bs, Lr, c, rd, ud, Hl, Hkl, G;
    int causal, mode, step, split, ring_rank_only;
    float scale_log2;  // softmax scale * log2(e)
    const int32_t *cu;  // packed samples, or nullptr
    uint32_t nseq;
    FastDiv f_Lr, f_bs, f_Hl, f_ud;
};

template <typename T, int EPL> struct Lane;
template <int EPL> struct Lane<float, EPL> {
    __device__ static void load(const float *p, float *x) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) x[i] = p[i];
    }
    __device__ static void store(float *p, const float *x) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) p[i] = x[i];
    }
};
template <int EPL> struct Lane<__nv_bfloat16, EPL> {
    __device__ static void load(const __nv_bfloat16 *p, float *x) {
#pragma unroll
        for (int i = 0; i < EPL; i += 2) {
            float2 f = bf16x2_to_float2(*reinterpret_cast<const uint32_t *>(p + i));
            x[i] = f.x;
            x[i + 1] = f.y;
        }
    }
    __device__ static void store(__nv_bfloat16 *p, const float *x) {
#pragma unroll
        for (int i = 0; i < EPL; i += 2) *reinterpret_cast<uint32_t *>(p + i) = float2_to_bf16x2(x[i], x[i + 1]);
    }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename T, int HD>
__global__ void __launch_bounds__(256) attn_simt_kernel(const AttnK p) {
    constexpr int EPL = HD / 32;
    const int lane = threadIdx.x & 31;
    const uint32_t row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= p.nrows) return;
    uint32_t t0, pq, b, h, u, r;
    p.f_Lr.divmod(row, t0, pq);
    p.f_bs.divmod(t0, t0, b);
    p.f_Hl.divmod(t0, t0, h);
    p.f_ud.divmod(t0, r, u);
    if (p.ring_rank_only > 0 && r != (uint32_t)(p.ring_rank_only - 1)) return;
    const int64_t qpos = split_pos(p.split, r, pq, p.c, p.rd);
    const uint32_t kh = h / p.G;
    // packed samples: the keys of the query's own sample [sa, se) only
    uint32_t sa = 0, se = p.Lr * p.rd;
    if (p.cu) sample_bounds(p.cu, p.nseq, (uint32_t)qpos, p.Lr * p.rd, sa, se);

    float qv[EPL], acc[EPL];
    Lane<T, EPL>::load(static_cast<const T *>(p.q) + (size_t)row * HD + lane * EPL, qv);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        qv[i] *= p.scale_log2;
        acc[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;  // running max (log2 domain) and normaliser

    const int t_begin = p.mode == USP_MODE_FUSED ? 0 : p.step;
    const int t_end = p.mode == USP_MODE_FUSED ? (int)p.rd : p.step + 1;
    for (int t = t_begin; t < t_end; ++t) {
        const uint32_t s = (r + p.rd - (uint32_t)t) % p.rd;
        // visible keys of rank s's block: a range of rows (every split's position map increases)
        const int64_t j0 = sa > 0 ? split_visible(p.split, (int64_t)sa - 1, s, p.c, p.rd) : 0;
        const int64_t nvis = p.causal ? split_visible(p.split, qpos, s, p.c, p.rd)
                                      : split_visible(p.split, (int64_t)se - 1, s, p.c, p.rd);
        const size_t kv_row0 = ((((size_t)s * p.ud + u) * p.Hkl + kh) * p.bs + b) * p.Lr;
        const T *kp = static_cast<const T *>(p.k) + kv_row0 * HD + lane * EPL;
        const T *vp = static_cast<const T *>(p.v) + kv_row0 * HD + lane * EPL;
        for (int64_t j = j0; j < nvis; ++j) {
            float kv[EPL], vv[EPL];
            Lane<T, EPL>::load(kp + j * HD, kv);
            Lane<T, EPL>::load(vp + j * HD, vv);
            float d = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) d = fmaf(qv[i], kv[i], d);
            const float sc = warp_sum(d);
            if (sc > m) {
                const float a = exp2f(m - sc);  // 0 when m = -inf
                l = l * a + 1.f;
#pragma unroll
                for (int i = 0; i < EPL; ++i) acc[i] = fmaf(acc[i], a, vv[i]);
                m = sc;
            } else {
                const float e = exp2f(sc - m);
                l += e;
#pragma unroll
                for (int i = 0; i < EPL; ++i) acc[i] = fmaf(e, vv[i], acc[i]);
            }
        }
    }
    float lse_row;
    if (l > 0.f) {
        const float inv = 1.f / l;
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[i] *= inv;
        lse_row = (m + log2f(l)) * 0.69314718055994531f;
    } else {
        lse_row = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
    }
    T *op = static_cast<T *>(p.out) + (size_t)row * HD + lane * EPL;
    if (p.mode == USP_MODE_ACCUM) {
        float prev[EPL], w1, w2, lm;
        Lane<T, EPL>::load(op, prev);
        merge_weights(p.lse[row], lse_row, w1, w2, lm);
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[i] = w1 * prev[i] + w2 * acc[i];
        lse_row = lm;
        __syncwarp();
    }
    Lane<T, EPL>::store(op, acc);
    if (lane == 0) p.lse[row] = lse_row;
}

template <typename T, int HD>
int launch_simt_typed(const AttnK &k, cudaStream_t s) {
    const uint32_t blocks = (k.nrows + 7) / 8;
    attn_simt_kernel<T, HD><<<blocks, 256, 0, s>>>(k);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace

int launch_attn_simt(const AttnArgs &a, cudaStream_t s) {
    AttnK k{};
    k.q = a.q; k.k = a.k; k.v = a.v; k.out = a.out; k.lse = a.lse;
    const int64_t nrows = (int64_t)a.hq * a.bs * a.L;
    if (nrows >= (int64_t(1) << 31)) return USP_ERR_UNSUPPORTED;
    k.nrows = (uint32_t)nrows;
    k.bs = (uint32_t)a.bs;
    k.rd = (uint32_t)a.rd;
    k.ud = (uint32_t)a.ud;
    k.Lr = (uint32_t)(a.L / a.rd);
    k.c = (uint32_t)(a.L / (2 * a.rd));
    k.Hl = (uint32_t)(a.hq / a.ud);
    k.Hkl = (uint32_t)heads_per_rank(a.hkv, a.ud);
    k.G = (uint32_t)(a.hq / a.hkv);
    k.causal = a.causal;
    k.mode = a.mode;
    k.step = a.step;
    k.split = a.split;
    k.ring_rank_only = a.ring_rank_only;
    k.scale_log2 = a.scale * 1.4426950408889634f;
    k.cu = a.cu;
    k.nseq = (uint32_t)a.nseq;
    k.f_Lr = FastDiv(k.Lr);
    k.f_bs = FastDiv(k.bs);
    k.f_Hl = FastDiv(k.Hl);
    k.f_ud = FastDiv(k.ud);
    if (a.dtype == USP_F32) {
        return a.hd == 64 ? launch_simt_typed<float, 64>(k, s) : launch_simt_typed<float, 128>(k, s);
    }
    return a.hd == 64 ? launch_simt_typed<__nv_bfloat16, 64>(k, s) : launch_simt_typed<__nv_bfloat16, 128>(k, s);
}

}  // namespace usp
