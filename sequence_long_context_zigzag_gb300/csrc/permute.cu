// permute.cu -- the zigzag split (Algorithm 2 of the USP review) and AllToAll4D (its section 三) as
// on-device row gathers. A "row" is the hd contiguous elements of one (token, head); every mode is a
// bijection between rows, so the kernel maps row indices and copies rows bit-exactly.
//
// Modes: the split (natural -> local) and its inverse, the all-to-all (local -> head-sharded) and its
// inverse, and the two composed in one pass (natural -> head-sharded and back). Composing them gives
// a direct map: row p of ring rank r in the head-sharded layout is global token zig(r, p), because
// the all-to-all concatenates the Ulysses ranks' pieces in rank order, which is exactly the
// ring-local sequence Algorithm 2 chunked. The composed pass reads and writes each tensor once. The
// zigzag split is the default; the plain ring's contiguous split and the round-robin stripe split
// use the same kernel with another position map. A forward all-to-all of fewer heads than Ulysses
// ranks (K/V of GQA/MQA, hkv < ud) replicates: rank u' receives head u' / (ud / H), the one its query
// heads read (the USP review's section 三 lists K/V head counts unlike Q's among AllToAll4D's duties).
//
// Work split: one warp owns a batch of 32 logical rows. Lane l computes the source and destination
// row of row l of the batch (integer index math with multiply-high division), publishes them in
// shared memory, then the warp copies the whole batch with lane-consecutive 16-byte vectors (4-byte
// words for rows that are not a multiple of 16 bytes, such as lse), so each load and store
// instruction covers contiguous row segments (a 256-byte row is one half-warp). Loads are issued in
// groups of 8 before their stores to keep enough bytes in flight for HBM. Up to four tensors (e.g.
// Q, K and V, or out and lse) share one launch; batches are numbered across them, and each tensor
// has its own row size.
#include "usp_device.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

struct PermJobK {
    const char *src;
    char *dst;
    uint32_t nrows, batch0;  // logical rows; first warp batch of this tensor
    uint32_t H, Ht, h0, Hl;
    uint32_t vec16, vpr;       // copy units: 16-byte vectors (vec16) or 4-byte words; units per row
    FastDiv f_H, f_Hl, f_rep;  // f_rep: ranks sharing one head (1 unless H < ud in a forward a2a)
    FastDiv f_vpr;
};

struct PermK {
    int mode, split, njobs;
    PermJobK job[kMaxPermJobs];
    uint32_t nbatch;  // total warp batches over all tensors
    uint32_t bs, L, rd, ud, Lu, Lr, c;
    int r_fixed, u_fixed;
    FastDiv f_Lu, f_bs, f_ud, f_Lr;
};

// map logical row i of tensor j to (source row, destination row) in units of rows
__device__ __forceinline__ void map_row(const PermK &p, const PermJobK &jb, uint32_t i, int64_t &srow,
                                        int64_t &drow) {
    uint32_t q;
    if (p.mode == PERM_EXTRACT || p.mode == PERM_EXTRACT_INV) {
        // logical order = local layout [rd][ud][bs][Lu][H] (or [bs][Lu][H] for one rank)
        uint32_t h, j, b, u, r;
        jb.f_H.divmod(i, q, h);
        p.f_Lu.divmod(q, q, j);
        p.f_bs.divmod(q, q, b);
        if (p.r_fixed >= 0) {
            r = (uint32_t)p.r_fixed;
            u = (uint32_t)p.u_fixed;
        } else {
            p.f_ud.divmod(q, r, u);
        }
        const int64_t g = split_pos(p.split, r, (int64_t)u * p.Lu + j, p.c, p.rd);
        const int64_t nat = ((int64_t)b * p.L + g) * jb.Ht + jb.h0 + h;
        if (p.mode == PERM_EXTRACT) { srow = nat; drow = i; }
        else { srow = i; drow = nat; }
    } else if (p.mode == PERM_A2A_FWD || p.mode == PERM_FUSED_FWD || p.mode == PERM_FUSED_INV) {
        // logical order = head-sharded layout [rd][ud'][Hl][bs][Lr]
        uint32_t pp, b, hl, up, r;
        p.f_Lr.divmod(i, q, pp);
        p.f_bs.divmod(q, q, b);
        jb.f_Hl.divmod(q, q, hl);
        p.f_ud.divmod(q, r, up);
        const int64_t head = (int64_t)jb.h0 + (int64_t)jb.f_rep.div(up) * jb.Hl + hl;
        if (p.mode == PERM_A2A_FWD) {
            uint32_t u, j;
            p.f_Lu.divmod(pp, u, j);
            srow = ((((int64_t)r * p.ud + u) * p.bs + b) * p.Lu + j) * jb.Ht + head;
            drow = i;
        } else {
            const int64_t nat = ((int64_t)b * p.L + split_pos(p.split, r, pp, p.c, p.rd)) * jb.Ht + head;
            if (p.mode == PERM_FUSED_FWD) { srow = nat; drow = i; }
            else { srow = i; drow = nat; }
        }
    } else {
        // PERM_A2A_INV: logical order = sequence-sharded layout [rd][ud][bs][Lu][H]
        uint32_t h, j, b, u, r, us, hl;
        jb.f_H.divmod(i, q, h);
        p.f_Lu.divmod(q, q, j);
        p.f_bs.divmod(q, q, b);
        p.f_ud.divmod(q, r, u);
        jb.f_Hl.divmod(h, us, hl);
        srow = ((((int64_t)r * p.ud + us) * jb.Hl + hl) * p.bs + b) * p.Lr + (int64_t)u * p.Lu + j;
        drow = ((((int64_t)r * p.ud + u) * p.bs + b) * p.Lu + j) * jb.Ht + jb.h0 + h;
    }
}

template <typename T>
__device__ __forceinline__ T load_stream(const T *p) { return __ldcs(p); }

constexpr int kWarps = 8;
constexpr int kGroup = 8;

// the warp's batch of rows_here rows, in units U (uint4: 16-byte vectors, unsigned int: 4-byte words)
template <typename U>
__device__ __forceinline__ void copy_batch(const PermJobK &jb, const int64_t *s_src, const int64_t *s_dst,
                                           uint32_t rows_here, int lane) {
    const uint32_t units_here = rows_here * jb.vpr;
    const U *src = reinterpret_cast<const U *>(jb.src);
    U *dst = reinterpret_cast<U *>(jb.dst);
    for (uint32_t base = 0; base < units_here; base += 32 * kGroup) {
        U buf[kGroup];
        int64_t doff[kGroup];
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            const uint32_t v = base + k * 32 + lane;
            doff[k] = -1;
            if (v < units_here) {
                uint32_t rr, col;
                jb.f_vpr.divmod(v, rr, col);
                buf[k] = load_stream(src + s_src[rr] * jb.vpr + col);
                doff[k] = s_dst[rr] * jb.vpr + col;
            }
        }
#pragma unroll
        for (int k = 0; k < kGroup; ++k)
            if (doff[k] >= 0) dst[doff[k]] = buf[k];
    }
}

__global__ void __launch_bounds__(kWarps * 32) permute_rows_kernel(const __grid_constant__ PermK p) {
    __shared__ int64_t s_src[kWarps][32];
    __shared__ int64_t s_dst[kWarps][32];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    for (uint32_t batch = blockIdx.x * kWarps + w; batch < p.nbatch; batch += gridDim.x * kWarps) {
        int jx = 0;
#pragma unroll
        for (int k = 1; k < kMaxPermJobs; ++k)
            if (k < p.njobs && batch >= p.job[k].batch0) jx = k;
        const PermJobK &jb = p.job[jx];
        const uint32_t row0 = (batch - jb.batch0) * 32;
        const uint32_t i = row0 + lane;
        int64_t sr = -1, dr = -1;
        if (i < jb.nrows) map_row(p, jb, i, sr, dr);
        __syncwarp();
        s_src[w][lane] = sr;
        s_dst[w][lane] = dr;
        __syncwarp();
        const uint32_t rows_here = min(32u, jb.nrows - row0);
        if (jb.vec16) copy_batch<uint4>(jb, s_src[w], s_dst[w], rows_here, lane);
        else copy_batch<unsigned int>(jb, s_src[w], s_dst[w], rows_here, lane);
        __syncwarp();
    }
}

// ---- the adjoint of the replicating all-to-all: each head receives the sum of its replicas ----
// Destination rows are enumerated as [rd][Lr][bs][H] (ring rank, ring-local row, batch, head); row
// (r, p, b, h) is natural token split_pos(r, p) (fused inverse) or sequence-sharded slot
// (r, p / Lu, b, p % Lu) (plain inverse), and sums head-sharded rows (r, u', 0, b, p) over the
// replicas u' in [h rep, (h + 1) rep). One thread per 16-byte vector; fp32 sums, rounded once.
struct RepSumK {
    const char *src;
    char *dst;
    uint32_t nvec;  // destination rows x vectors per row
    uint32_t Ht, h0, rep, bs, L, Lr, Lu, c, rd, ud, vpr;
    int mode, split;
    FastDiv f_H, f_bs, f_Lr, f_Lu, f_vpr;
};

__device__ __forceinline__ void add_vec(float (&acc)[8], uint4 w, bool bf16) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    if (bf16) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = bf16x2_to_float2(u[e]);
            acc[2 * e] += f.x;
            acc[2 * e + 1] += f.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += __uint_as_float(u[e]);
    }
}

__global__ void __launch_bounds__(256) replica_sum_kernel(const __grid_constant__ RepSumK p, int bf16) {
    for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < p.nvec; t += gridDim.x * blockDim.x) {
        uint32_t row, vec, q, h, b, pp, r;
        p.f_vpr.divmod(t, row, vec);
        p.f_H.divmod(row, q, h);
        p.f_bs.divmod(q, q, b);
        p.f_Lr.divmod(q, r, pp);
        int64_t drow;
        if (p.mode == PERM_FUSED_INV) {
            drow = ((int64_t)b * p.L + split_pos(p.split, r, pp, p.c, p.rd)) * p.Ht + p.h0 + h;
        } else {
            uint32_t u, j;
            p.f_Lu.divmod(pp, u, j);
            drow = ((((int64_t)r * p.ud + u) * p.bs + b) * p.Lu + j) * p.Ht + p.h0 + h;
        }
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (uint32_t k = 0; k < p.rep; ++k) {
            const int64_t srow = (((int64_t)r * p.ud + h * p.rep + k) * p.bs + b) * p.Lr + pp;
            add_vec(acc, __ldg(reinterpret_cast<const uint4 *>(p.src) + srow * p.vpr + vec), bf16 != 0);
        }
        uint4 o;
        if (bf16) {
            o = make_uint4(float2_to_bf16x2(acc[0], acc[1]), float2_to_bf16x2(acc[2], acc[3]),
                           float2_to_bf16x2(acc[4], acc[5]), float2_to_bf16x2(acc[6], acc[7]));
        } else {
            o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                           __float_as_uint(acc[3]));
        }
        reinterpret_cast<uint4 *>(p.dst)[drow * p.vpr + vec] = o;
    }
}

int launch_replica_sum(const PermArgs &a, const PermJob &j, int sms, cudaStream_t s) {
    if (j.row_bytes % 16 != 0 || (j.dtype != USP_BF16 && j.dtype != USP_F32)) return USP_ERR_UNSUPPORTED;
    RepSumK p{};
    p.src = j.src;
    p.dst = j.dst;
    p.mode = a.mode;
    p.split = a.split;
    p.Ht = (uint32_t)j.H_total;
    p.h0 = (uint32_t)j.h0;
    p.rep = (uint32_t)(a.ud / j.H);
    p.bs = (uint32_t)a.bs;
    p.L = (uint32_t)a.L;
    p.rd = (uint32_t)a.rd;
    p.ud = (uint32_t)a.ud;
    p.Lr = (uint32_t)(a.L / a.rd);
    p.Lu = p.Lr / p.ud;
    p.c = (uint32_t)(a.L / (2 * a.rd));
    p.vpr = (uint32_t)(j.row_bytes / 16);
    const int64_t nvec = (int64_t)a.rd * p.Lr * a.bs * j.H * p.vpr;
    if (nvec == 0) return USP_OK;
    if (nvec >= (int64_t(1) << 31)) return USP_ERR_UNSUPPORTED;
    p.nvec = (uint32_t)nvec;
    p.f_H = FastDiv((uint32_t)j.H);
    p.f_bs = FastDiv(p.bs);
    p.f_Lr = FastDiv(p.Lr);
    p.f_Lu = FastDiv(p.Lu);
    p.f_vpr = FastDiv(p.vpr);
    int64_t blocks = (nvec + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    replica_sum_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, j.dtype == USP_BF16 ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace

int launch_permute(const PermArgs &a, cudaStream_t s) {
    const DeviceInfo *di = device_info();
    if (!di) return USP_ERR_CUDA;
    if (a.njobs < 1 || a.njobs > kMaxPermJobs) return USP_ERR_INVALID_ARG;
    // inverse all-to-all of replicated heads (H < ud): the replica sum, one launch per such tensor;
    // the other tensors go through the row gather below
    if (a.mode == PERM_A2A_INV || a.mode == PERM_FUSED_INV) {
        PermArgs rest = a;
        rest.njobs = 0;
        for (int k = 0; k < a.njobs; ++k) {
            if (a.job[k].H > 0 && a.job[k].H < a.ud) {
                const int rc = launch_replica_sum(a, a.job[k], di->sm_count, s);
                if (rc) return rc;
            } else {
                rest.job[rest.njobs++] = a.job[k];
            }
        }
        if (rest.njobs == 0) return USP_OK;
        if (rest.njobs < a.njobs) return launch_permute(rest, s);
    }
    PermK p{};
    p.mode = a.mode;
    p.split = a.split;
    p.njobs = a.njobs;
    p.bs = (uint32_t)a.bs;
    p.L = (uint32_t)a.L;
    p.rd = (uint32_t)a.rd;
    p.ud = (uint32_t)a.ud;
    p.Lr = (uint32_t)(a.L / a.rd);
    p.Lu = p.Lr / p.ud;
    p.c = (uint32_t)(a.L / (2 * a.rd));
    p.r_fixed = a.r_fixed;
    p.u_fixed = a.u_fixed;
    const int64_t ranks = (a.r_fixed >= 0) ? 1 : (int64_t)a.rd * a.ud;
    const bool to_heads = a.mode == PERM_A2A_FWD || a.mode == PERM_FUSED_FWD;
    int64_t nbatch = 0;
    for (int k = 0; k < a.njobs; ++k) {
        const PermJob &j = a.job[k];
        PermJobK &jk = p.job[k];
        jk.src = j.src;
        jk.dst = j.dst;
        jk.H = (uint32_t)j.H;
        const bool vec16 = (j.row_bytes % 16) == 0;
        const int64_t vpr = j.row_bytes / (vec16 ? 16 : 4);
        if (vpr < 1 || 32 * vpr >= (int64_t(1) << 31)) return USP_ERR_UNSUPPORTED;
        jk.vec16 = vec16 ? 1u : 0u;
        jk.vpr = (uint32_t)vpr;
        jk.f_vpr = FastDiv(jk.vpr);
        jk.Ht = (uint32_t)j.H_total;
        jk.h0 = (uint32_t)j.h0;
        // a forward all-to-all of fewer heads than Ulysses ranks replicates: one head per rank
        const bool rep = to_heads && jk.H > 0 && jk.H < p.ud;
        jk.Hl = rep ? 1 : jk.H / p.ud;
        jk.f_H = FastDiv(jk.H ? jk.H : 1);
        jk.f_Hl = FastDiv(jk.Hl ? jk.Hl : 1);
        jk.f_rep = FastDiv(rep ? p.ud / jk.H : 1);
        // rows of the destination (= of the source, except when replicating)
        const int64_t rows_per_tok = rep ? (int64_t)p.ud : (int64_t)j.H;
        const int64_t nrows = ranks * a.bs * (int64_t)p.Lu * rows_per_tok;
        if (nrows >= (int64_t(1) << 31)) return USP_ERR_UNSUPPORTED;
        jk.nrows = (uint32_t)nrows;
        jk.batch0 = (uint32_t)nbatch;
        nbatch += (nrows + 31) / 32;
    }
    if (nbatch == 0) return USP_OK;
    if (nbatch >= (int64_t(1) << 31)) return USP_ERR_UNSUPPORTED;
    p.nbatch = (uint32_t)nbatch;
    p.f_Lu = FastDiv(p.Lu);
    p.f_bs = FastDiv(p.bs);
    p.f_ud = FastDiv(p.ud);
    p.f_Lr = FastDiv(p.Lr);
    int64_t blocks = (nbatch + kWarps - 1) / kWarps;
    const int64_t cap = a.max_blocks > 0 ? (int64_t)a.max_blocks : (int64_t)di->sm_count * 8;
    if (blocks > cap) blocks = cap;
    permute_rows_kernel<<<(unsigned)blocks, kWarps * 32, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace usp
