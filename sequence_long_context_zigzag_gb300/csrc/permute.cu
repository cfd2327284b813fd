// permute.cu -- the zigzag split (Algorithm 2 of the USP review) and AllToAll4D (its section 三) as
// on-device row gathers. A "row" is the hd contiguous elements of one (token, head); every mode is a
// bijection between rows, so the kernel maps row indices and copies rows bit-exactly.
//
// Work split: one warp owns a batch of 32 logical rows. Lane l computes the source and destination
// row of row l of the batch (integer index math with multiply-high division), publishes them in
// shared memory, then the warp copies the whole batch with lane-consecutive 16-byte vectors, so each
// load and store instruction covers contiguous row segments (a 256-byte row is one half-warp).
// Loads are issued in groups of 8 before their stores to keep enough bytes in flight for HBM.
#include "usp_internal.cuh"

namespace usp {
namespace {

struct PermK {
    const char *src;
    char *dst;
    uint32_t nrows;  // logical rows iterated
    int mode;
    uint32_t bs, L, H, Ht, h0, rd, ud, Lu, Lr, c, Hl;
    int r_fixed, u_fixed;
    int64_t row_bytes;
    uint32_t vpr;  // units (16-byte vectors or 4-byte words) per row
    FastDiv f_vpr, f_H, f_Lu, f_bs, f_ud, f_Hl, f_Lr;
};

// map logical row i to (source row, destination row) in units of rows
__device__ __forceinline__ void map_row(const PermK &p, uint32_t i, int64_t &srow, int64_t &drow) {
    uint32_t q;
    if (p.mode == PERM_EXTRACT || p.mode == PERM_EXTRACT_INV) {
        // logical order = local layout [rd][ud][bs][Lu][H] (or [bs][Lu][H] for one rank)
        uint32_t h, j, b, u, r;
        p.f_H.divmod(i, q, h);
        p.f_Lu.divmod(q, q, j);
        p.f_bs.divmod(q, q, b);
        if (p.r_fixed >= 0) {
            r = (uint32_t)p.r_fixed;
            u = (uint32_t)p.u_fixed;
        } else {
            p.f_ud.divmod(q, r, u);
        }
        const int64_t g = zig_pos(r, (int64_t)u * p.Lu + j, p.c, p.rd);
        const int64_t nat = ((int64_t)b * p.L + g) * p.Ht + p.h0 + h;
        if (p.mode == PERM_EXTRACT) { srow = nat; drow = i; }
        else { srow = i; drow = nat; }
    } else if (p.mode == PERM_A2A_FWD) {
        // logical order = head-sharded layout [rd][ud'][Hl][bs][Lr]
        uint32_t pp, b, hl, up, r, u, j;
        p.f_Lr.divmod(i, q, pp);
        p.f_bs.divmod(q, q, b);
        p.f_Hl.divmod(q, q, hl);
        p.f_ud.divmod(q, r, up);
        p.f_Lu.divmod(pp, u, j);
        srow = ((((int64_t)r * p.ud + u) * p.bs + b) * p.Lu + j) * p.Ht + p.h0 + (int64_t)up * p.Hl + hl;
        drow = i;
    } else {
        // PERM_A2A_INV: logical order = sequence-sharded layout [rd][ud][bs][Lu][H]
        uint32_t h, j, b, u, r, us, hl;
        p.f_H.divmod(i, q, h);
        p.f_Lu.divmod(q, q, j);
        p.f_bs.divmod(q, q, b);
        p.f_ud.divmod(q, r, u);
        p.f_Hl.divmod(h, us, hl);
        srow = ((((int64_t)r * p.ud + us) * p.Hl + hl) * p.bs + b) * p.Lr + (int64_t)u * p.Lu + j;
        drow = ((((int64_t)r * p.ud + u) * p.bs + b) * p.Lu + j) * p.Ht + p.h0 + h;
    }
}

template <typename T>
__device__ __forceinline__ T load_stream(const T *p) { return __ldcs(p); }

constexpr int kWarps = 8;
constexpr int kGroup = 8;

template <typename T>  // T = uint4 (16-byte units) or unsigned int (4-byte units)
__global__ void __launch_bounds__(kWarps * 32) permute_rows_kernel(const PermK p) {
    __shared__ int64_t s_src[kWarps][32];
    __shared__ int64_t s_dst[kWarps][32];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const uint32_t nbatch = (p.nrows + 31) / 32;
    const uint32_t total_units = 32u * p.vpr;
    for (uint32_t batch = blockIdx.x * kWarps + w; batch < nbatch; batch += gridDim.x * kWarps) {
        const uint32_t row0 = batch * 32;
        const uint32_t i = row0 + lane;
        int64_t sr = -1, dr = -1;
        if (i < p.nrows) map_row(p, i, sr, dr);
        __syncwarp();
        s_src[w][lane] = sr;
        s_dst[w][lane] = dr;
        __syncwarp();
        const uint32_t rows_here = min(32u, p.nrows - row0);
        const uint32_t units_here = rows_here * p.vpr;
        for (uint32_t base = 0; base < total_units; base += 32 * kGroup) {
            T buf[kGroup];
            int64_t doff[kGroup];
#pragma unroll
            for (int k = 0; k < kGroup; ++k) {
                const uint32_t v = base + k * 32 + lane;
                doff[k] = -1;
                if (v < units_here) {
                    uint32_t rr, col;
                    p.f_vpr.divmod(v, rr, col);
                    const T *sp = reinterpret_cast<const T *>(p.src) + s_src[w][rr] * p.vpr + col;
                    buf[k] = load_stream(sp);
                    doff[k] = s_dst[w][rr] * p.vpr + col;
                }
            }
#pragma unroll
            for (int k = 0; k < kGroup; ++k)
                if (doff[k] >= 0) reinterpret_cast<T *>(p.dst)[doff[k]] = buf[k];
        }
        __syncwarp();
    }
}

}  // namespace

int launch_permute(const PermArgs &a, cudaStream_t s) {
    const DeviceInfo *di = device_info();
    if (!di) return USP_ERR_CUDA;
    PermK p{};
    p.src = a.src;
    p.dst = a.dst;
    p.mode = a.mode;
    p.bs = (uint32_t)a.bs;
    p.L = (uint32_t)a.L;
    p.H = (uint32_t)a.H;
    p.Ht = (uint32_t)a.H_total;
    p.h0 = (uint32_t)a.h0;
    p.rd = (uint32_t)a.rd;
    p.ud = (uint32_t)a.ud;
    p.Lr = (uint32_t)(a.L / a.rd);
    p.Lu = p.Lr / p.ud;
    p.c = (uint32_t)(a.L / (2 * a.rd));
    p.Hl = p.H / p.ud;
    p.r_fixed = a.r_fixed;
    p.u_fixed = a.u_fixed;
    p.row_bytes = a.row_bytes;
    const bool vec16 = (a.row_bytes % 16) == 0;
    p.vpr = (uint32_t)(a.row_bytes / (vec16 ? 16 : 4));
    const int64_t ranks = (a.r_fixed >= 0) ? 1 : (int64_t)a.rd * a.ud;
    const int64_t nrows = ranks * a.bs * (int64_t)p.Lu * a.H;  // same count in every mode
    if (nrows <= 0) return USP_OK;
    if (nrows >= (int64_t(1) << 31) || (int64_t)32 * p.vpr >= (int64_t(1) << 31)) return USP_ERR_UNSUPPORTED;
    p.nrows = (uint32_t)nrows;
    p.f_vpr = FastDiv(p.vpr);
    p.f_H = FastDiv(p.H);
    p.f_Lu = FastDiv(p.Lu);
    p.f_bs = FastDiv(p.bs);
    p.f_ud = FastDiv(p.ud);
    p.f_Hl = FastDiv(p.Hl ? p.Hl : 1);
    p.f_Lr = FastDiv(p.Lr);
    const int64_t nbatch = (nrows + 31) / 32;
    int64_t blocks = (nbatch + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)di->sm_count * 8;
    if (blocks > cap) blocks = cap;
    if (vec16)
        permute_rows_kernel<uint4><<<(unsigned)blocks, kWarps * 32, 0, s>>>(p);
    else
        permute_rows_kernel<unsigned int><<<(unsigned)blocks, kWarps * 32, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace usp
