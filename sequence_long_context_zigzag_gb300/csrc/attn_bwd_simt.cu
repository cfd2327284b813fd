// attn_bwd_simt.cu -- ring attention backward on the CUDA cores (fp32 arithmetic), and the row dot
// product D_i = <dout_i, out_i> it needs.
//
// The gradients are those of the forward (chain rule through softmax): with P_ij = exp(s_ij - lse_i)
// from the forward's final lse, dP_ij = <dout_i, v_j> and dS_ij = P_ij (dP_ij - D_i),
//   dq_i = scale sum_j dS_ij k_j,   dk_j = scale sum_i dS_ij q_i,   dv_j = sum_i P_ij dout_i,
// over the forward's causal (query, key) pairs. Two kernels, one warp per output row each:
//   * dq: a query row of ring rank r walks the ring in the Context-Parallel page's Fig. 1 order
//     (step t: KV block of rank (r - t) mod rd), its visible keys being a range of each block's rows
//     (a prefix of it unless samples are packed);
//   * dk/dv: a key row of rank s meets the queries of every ring rank once; those that see it are a
//     range of each rank's rows (every split's position map increases with the row; a suffix unless
//     samples are packed), and the query heads of its group (or, for a replicated KV head, all of the
//     rank's query heads) add up.
// In a multi-GPU ring the dk/dv partials would travel with the KV block and be home after rd steps;
// here each key row's warp forms its whole sum.
#include <math.h>

#include "usp_device.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

struct BwdK {
    const void *q, *k, *v, *dout;
    const float *lse, *delta;
    void *dq, *dk, *dv;
    uint32_t nq_rows, nkv_rows, bs, Lr, c, rd, ud, Hl, Hkl, G;
    int causal, split;
    float scale, scale_log2;
    const int32_t *cu;  // packed samples, or nullptr
    uint32_t nseq;
    FastDiv f_Lr, f_bs, f_Hl, f_Hkl, f_ud;
};

// number of rank-s rows whose global position is below x (a prefix of the block)
__device__ __forceinline__ int64_t rows_before(int split, int64_t x, int64_t s, int64_t c, int64_t rd) {
    return x > 0 ? split_visible(split, x - 1, s, c, rd) : 0;
}

constexpr float kLog2e = 1.4426950408889634f;

template <typename T, int EPL> struct Row;
template <int EPL> struct Row<float, EPL> {
    __device__ static void load(const float *p, float *x) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) x[i] = p[i];
    }
    __device__ static void store(float *p, const float *x) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) p[i] = x[i];
    }
};
template <int EPL> struct Row<__nv_bfloat16, EPL> {
    __device__ static void load(const __nv_bfloat16 *p, float *x) {
#pragma unroll
        for (int i = 0; i < EPL; i += 2) {
            const float2 f = bf16x2_to_float2(*reinterpret_cast<const uint32_t *>(p + i));
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
__global__ void __launch_bounds__(256) bwd_dq_kernel(const BwdK p) {
    constexpr int EPL = HD / 32;
    const int lane = threadIdx.x & 31;
    const uint32_t row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= p.nq_rows) return;
    uint32_t t0, pq, b, h, u, r;
    p.f_Lr.divmod(row, t0, pq);
    p.f_bs.divmod(t0, t0, b);
    p.f_Hl.divmod(t0, t0, h);
    p.f_ud.divmod(t0, r, u);
    const int64_t qpos = split_pos(p.split, r, pq, p.c, p.rd);
    const uint32_t kh = h / p.G;
    uint32_t sa = 0, se = p.Lr * p.rd;  // the row's sample (packed sequences)
    if (p.cu) sample_bounds(p.cu, p.nseq, (uint32_t)qpos, p.Lr * p.rd, sa, se);
    float qv[EPL], gv[EPL], acc[EPL];
    Row<T, EPL>::load(static_cast<const T *>(p.q) + (size_t)row * HD + lane * EPL, qv);
    Row<T, EPL>::load(static_cast<const T *>(p.dout) + (size_t)row * HD + lane * EPL, gv);
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
    const float lse2 = p.lse[row] * kLog2e, Di = p.delta[row];
    for (uint32_t t = 0; t < p.rd; ++t) {
        const uint32_t s = (r + p.rd - t) % p.rd;
        const int64_t j0 = rows_before(p.split, sa, s, p.c, p.rd);
        const int64_t nvis = p.causal ? split_visible(p.split, qpos, s, p.c, p.rd)
                                      : rows_before(p.split, se, s, p.c, p.rd);
        const size_t kv_row0 = ((((size_t)s * p.ud + u) * p.Hkl + kh) * p.bs + b) * p.Lr;
        const T *kp = static_cast<const T *>(p.k) + kv_row0 * HD + lane * EPL;
        const T *vp = static_cast<const T *>(p.v) + kv_row0 * HD + lane * EPL;
        for (int64_t j = j0; j < nvis; ++j) {
            float kv[EPL], vv[EPL];
            Row<T, EPL>::load(kp + j * HD, kv);
            Row<T, EPL>::load(vp + j * HD, vv);
            float d = 0.f, e = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                d = fmaf(qv[i], kv[i], d);
                e = fmaf(gv[i], vv[i], e);
            }
            const float sc = warp_sum(d), dp = warp_sum(e);
            const float pr = exp2f(sc * p.scale_log2 - lse2);
            const float ds = pr * (dp - Di);
#pragma unroll
            for (int i = 0; i < EPL; ++i) acc[i] = fmaf(ds, kv[i], acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] *= p.scale;
    Row<T, EPL>::store(static_cast<T *>(p.dq) + (size_t)row * HD + lane * EPL, acc);
}

template <typename T, int HD>
__global__ void __launch_bounds__(256) bwd_dkv_kernel(const BwdK p) {
    constexpr int EPL = HD / 32;
    const int lane = threadIdx.x & 31;
    const uint32_t row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= p.nkv_rows) return;
    uint32_t t0, pk, b, kh, u, s;
    p.f_Lr.divmod(row, t0, pk);
    p.f_bs.divmod(t0, t0, b);
    p.f_Hkl.divmod(t0, t0, kh);
    p.f_ud.divmod(t0, s, u);
    const int64_t kpos = split_pos(p.split, s, pk, p.c, p.rd);
    uint32_t sa = 0, se = p.Lr * p.rd;  // the key's sample (packed sequences)
    if (p.cu) sample_bounds(p.cu, p.nseq, (uint32_t)kpos, p.Lr * p.rd, sa, se);
    float kv[EPL], vv[EPL], ak[EPL], av[EPL];
    Row<T, EPL>::load(static_cast<const T *>(p.k) + (size_t)row * HD + lane * EPL, kv);
    Row<T, EPL>::load(static_cast<const T *>(p.v) + (size_t)row * HD + lane * EPL, vv);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        ak[i] = 0.f;
        av[i] = 0.f;
    }
    // the rank's query heads that read this KV head: [kh G, kh G + G), clipped to the rank's Hl
    const uint32_t h_end = min(kh * p.G + p.G, p.Hl);
    for (uint32_t r = 0; r < p.rd; ++r) {
        // queries of rank r that see key position kpos: positions in [kpos, se) (causal) or [sa, se)
        // of the key's sample -- a range of rows
        const int64_t i0 = rows_before(p.split, p.causal ? kpos : (int64_t)sa, r, p.c, p.rd);
        const int64_t i1 = rows_before(p.split, se, r, p.c, p.rd);
        for (uint32_t h = kh * p.G; h < h_end; ++h) {
            const size_t q_row0 = ((((size_t)r * p.ud + u) * p.Hl + h) * p.bs + b) * p.Lr;
            const T *qp = static_cast<const T *>(p.q) + q_row0 * HD + lane * EPL;
            const T *gp = static_cast<const T *>(p.dout) + q_row0 * HD + lane * EPL;
            for (int64_t i = i0; i < i1; ++i) {
                float qv[EPL], gv[EPL];
                Row<T, EPL>::load(qp + i * HD, qv);
                Row<T, EPL>::load(gp + i * HD, gv);
                float d = 0.f, e = 0.f;
#pragma unroll
                for (int x = 0; x < EPL; ++x) {
                    d = fmaf(qv[x], kv[x], d);
                    e = fmaf(gv[x], vv[x], e);
                }
                const float sc = warp_sum(d), dp = warp_sum(e);
                const float pr = exp2f(sc * p.scale_log2 - p.lse[q_row0 + i] * kLog2e);
                const float ds = pr * (dp - p.delta[q_row0 + i]);
#pragma unroll
                for (int x = 0; x < EPL; ++x) {
                    ak[x] = fmaf(ds, qv[x], ak[x]);
                    av[x] = fmaf(pr, gv[x], av[x]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) ak[i] *= p.scale;
    Row<T, EPL>::store(static_cast<T *>(p.dk) + (size_t)row * HD + lane * EPL, ak);
    Row<T, EPL>::store(static_cast<T *>(p.dv) + (size_t)row * HD + lane * EPL, av);
}

template <typename T, int HD>
int launch_typed(const BwdK &k, cudaStream_t s) {
    if (k.nq_rows) bwd_dq_kernel<T, HD><<<(k.nq_rows + 7) / 8, 256, 0, s>>>(k);
    if (k.nkv_rows) bwd_dkv_kernel<T, HD><<<(k.nkv_rows + 7) / 8, 256, 0, s>>>(k);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

// D = <x_row, y_row> in fp32: one warp per row, 16-byte vectors, grid-stride over rows
template <typename T>
__global__ void __launch_bounds__(256) row_dot_kernel(const T *x, const T *y, float *out, int64_t rows, int vpr) {
    constexpr int EPV = 16 / sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * 8;
    for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < rows; r += warps) {
        float acc = 0.f;
        for (int v = lane; v < vpr; v += 32) {
            float a[EPV], b[EPV];
            Row<T, EPV>::load(x + (r * vpr + v) * EPV, a);
            Row<T, EPV>::load(y + (r * vpr + v) * EPV, b);
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc = fmaf(a[e], b[e], acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) out[r] = acc;
    }
}

}  // namespace

int launch_attn_bwd_simt(const BwdArgs &a, cudaStream_t s) {
    const AttnArgs &f = a.f;
    BwdK k{};
    k.q = f.q; k.k = f.k; k.v = f.v; k.dout = a.dout;
    k.lse = f.lse; k.delta = a.delta;
    k.dq = a.dq; k.dk = a.dk; k.dv = a.dv;
    k.bs = (uint32_t)f.bs;
    k.rd = (uint32_t)f.rd;
    k.ud = (uint32_t)f.ud;
    k.Lr = (uint32_t)(f.L / f.rd);
    k.c = (uint32_t)(f.L / (2 * f.rd));
    k.Hl = (uint32_t)(f.hq / f.ud);
    k.Hkl = (uint32_t)heads_per_rank(f.hkv, f.ud);
    k.G = (uint32_t)(f.hq / f.hkv);
    const int64_t nq = (int64_t)f.hq * f.bs * f.L;
    const int64_t nkv = (int64_t)k.Hkl * f.ud * f.bs * f.L;
    if (nq >= (int64_t(1) << 31) || nkv >= (int64_t(1) << 31)) return USP_ERR_UNSUPPORTED;
    k.nq_rows = (uint32_t)nq;
    k.nkv_rows = (uint32_t)nkv;
    k.causal = f.causal;
    k.split = f.split;
    k.scale = f.scale;
    k.scale_log2 = f.scale * kLog2e;
    k.cu = f.cu;
    k.nseq = (uint32_t)f.nseq;
    k.f_Lr = FastDiv(k.Lr);
    k.f_bs = FastDiv(k.bs);
    k.f_Hl = FastDiv(k.Hl);
    k.f_Hkl = FastDiv(k.Hkl);
    k.f_ud = FastDiv(k.ud);
    if (f.dtype == USP_F32)
        return f.hd == 64 ? launch_typed<float, 64>(k, s) : launch_typed<float, 128>(k, s);
    return f.hd == 64 ? launch_typed<__nv_bfloat16, 64>(k, s) : launch_typed<__nv_bfloat16, 128>(k, s);
}

int launch_row_dot(const void *x, const void *y, float *out, int64_t rows, int hd, int dtype, cudaStream_t s) {
    const DeviceInfo *di = device_info();
    if (!di) return USP_ERR_CUDA;
    const int vpr = hd * elem_size(dtype) / 16;
    int64_t blocks = (rows + 7) / 8;
    if (blocks > (int64_t)di->sm_count * 16) blocks = (int64_t)di->sm_count * 16;
    if (dtype == USP_F32)
        row_dot_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const float *>(x),
                                                                static_cast<const float *>(y), out, rows, vpr);
    else
        row_dot_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(y), out, rows, vpr);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace usp
