// usp_api.cu -- argument validation and dispatch for the C ABI declared in include/usp.h.
#include <math.h>
#include <mutex>

#include "tc_ptx.cuh"
#include "usp_internal.cuh"

// One status word per device: kernels whose bounded waits run out write a nonzero code here.
static __device__ int g_usp_status;

namespace usp {

static constexpr int kMaxDevices = 64;
static DeviceInfo g_info[kMaxDevices];
static bool g_info_ok[kMaxDevices];
static std::mutex g_info_mu;

const DeviceInfo *device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_info_mu);
    if (!g_info_ok[dev]) {
        DeviceInfo di{};
        if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        // the symbol's device address for the current device (host code cannot name it directly)
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&di.status), g_usp_status) != cudaSuccess)
            return nullptr;
        g_info[dev] = di;
        g_info_ok[dev] = true;
    }
    return &g_info[dev];
}

static bool overflow31(int64_t x) { return x < 0 || x >= (int64_t(1) << 31); }

// shared checks of a permute's dims. need_head_split: 0 = none (split only), 1 = ud must divide H,
// 2 = ud divides H or H divides ud (the all-to-all replicates heads, its inverse sums the replicas)
static int check_dims(const usp_dims &d, int need_head_split) {
    if (d.bs < 0 || d.L < 0 || d.H < 0 || d.hd <= 0 || d.rd <= 0 || d.ud <= 0 || d.h0 < 0 ||
        d.H_total < 0)
        return USP_ERR_INVALID_ARG;
    if (elem_size(d.dtype) == 0) return USP_ERR_DTYPE;
    if (d.split < USP_SPLIT_ZIGZAG || d.split > USP_SPLIT_STRIPE) return USP_ERR_INVALID_ARG;
    if (d.L % (2 * (int64_t)d.rd) != 0) return USP_ERR_SHAPE;
    if ((d.L / d.rd) % d.ud != 0) return USP_ERR_SHAPE;
    int32_t Ht = d.H_total ? d.H_total : d.H;
    if ((int64_t)d.h0 + d.H > Ht) return USP_ERR_SHAPE;
    if (need_head_split == 1 && d.H % d.ud != 0) return USP_ERR_SHAPE;
    if (need_head_split == 2 && d.H > 0 && heads_per_rank(d.H, d.ud) == 0) return USP_ERR_SHAPE;
    if (overflow31(d.bs * d.L * (int64_t)Ht) || overflow31(d.L) ||
        overflow31((int64_t)d.hd * elem_size(d.dtype)))
        return USP_ERR_UNSUPPORTED;
    return USP_OK;
}

static int check_ptr_align(const void *a, const void *b, int64_t row_bytes) {
    uintptr_t al = (row_bytes % 16 == 0) ? 16 : 4;
    if (row_bytes % 4 != 0) return USP_ERR_UNSUPPORTED;
    if (!aligned(a, al) || !aligned(b, al)) return USP_ERR_ALIGN;
    return USP_OK;
}

namespace {
// one thread waits (bounded) on an mbarrier that nothing arrives on: the wait runs out and records
// USP_ERR_TIMEOUT, exactly as a stalled wait inside the attention kernels would
__global__ void selftest_timeout_kernel(int *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t b = tc::smem_u32(&bar);
        tc::mbar_init(b, 1);
        tc::fence_barrier_init();
        tc::mbar_wait(b, 0, status, USP_ERR_TIMEOUT, limit_ns);
    }
}
}  // namespace

}  // namespace usp

using namespace usp;

extern "C" {

int usp_version(void) { return (1 << 16) | 0; }

const char *usp_strerror(int status) {
    switch (status) {
        case USP_OK: return "success";
        case USP_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or bad enum)";
        case USP_ERR_SHAPE: return "shape not divisible (L % 2rd, (L/rd) % ud, hq % ud, hq % hkv, hkv vs ud)";
        case USP_ERR_DTYPE: return "unknown dtype code";
        case USP_ERR_ALIGN: return "pointer not aligned as required";
        case USP_ERR_UNSUPPORTED: return "unsupported configuration";
        case USP_ERR_CUDA: return "CUDA runtime error";
        case USP_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        default: return "unknown status";
    }
}

int usp_extract_local(const void *src, void *dst, usp_dims d, int vr, int inverse, usp_stream_t stream) {
    int rc = check_dims(d, 0);
    if (rc) return rc;
    if (vr < -1 || vr >= d.rd * d.ud) return USP_ERR_INVALID_ARG;
    if (d.bs == 0 || d.L == 0 || d.H == 0) return USP_OK;
    if (!src || !dst) return USP_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)d.hd * elem_size(d.dtype);
    if ((rc = check_ptr_align(src, dst, row_bytes))) return rc;
    PermArgs a{};
    a.njobs = 1;
    a.job[0] = PermJob{static_cast<const char *>(src), static_cast<char *>(dst), d.H, d.H_total ? d.H_total : d.H,
                       d.h0, row_bytes, d.dtype};
    a.mode = inverse ? PERM_EXTRACT_INV : PERM_EXTRACT;
    a.split = d.split;
    a.bs = d.bs; a.L = d.L;
    a.rd = d.rd; a.ud = d.ud;
    a.r_fixed = vr >= 0 ? vr / d.ud : -1;
    a.u_fixed = vr >= 0 ? vr % d.ud : -1;
    return launch_permute(a, reinterpret_cast<cudaStream_t>(stream));
}

int usp_a2a4d(const void *src, void *dst, usp_dims d, int dir, usp_stream_t stream) {
    if (dir != 1 && dir != -1) return USP_ERR_INVALID_ARG;
    int rc = check_dims(d, 2);  // fewer heads than ranks: replicate (dir +1) or sum replicas (dir -1)
    if (rc) return rc;
    if (d.bs == 0 || d.L == 0 || d.H == 0) return USP_OK;
    if (!src || !dst) return USP_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)d.hd * elem_size(d.dtype);
    if ((rc = check_ptr_align(src, dst, row_bytes))) return rc;
    PermArgs a{};
    a.njobs = 1;
    a.job[0] = PermJob{static_cast<const char *>(src), static_cast<char *>(dst), d.H, d.H_total ? d.H_total : d.H,
                       d.h0, row_bytes, d.dtype};
    a.mode = dir > 0 ? PERM_A2A_FWD : PERM_A2A_INV;
    a.bs = d.bs; a.L = d.L;
    a.rd = d.rd; a.ud = d.ud;
    a.r_fixed = -1; a.u_fixed = -1;
    return launch_permute(a, reinterpret_cast<cudaStream_t>(stream));
}

// the multi-tensor permutes: usp_extract_a2a (split + all-to-all composed) and usp_a2a4d_multi
static int permute_multi(int n, const void *const *src, void *const *dst, const usp_dims *d, int mode,
                         usp_stream_t stream, int max_blocks = 0) {
    if (n < 1 || n > kMaxPermJobs || !src || !dst || !d) return USP_ERR_INVALID_ARG;
    PermArgs a{};
    a.njobs = n;
    a.mode = mode;
    a.r_fixed = -1;
    a.u_fixed = -1;
    int64_t work = 0;
    for (int k = 0; k < n; ++k) {
        const usp_dims &dk = d[k];
        int rc = check_dims(dk, 2);
        if (rc) return rc;
        // the split matters only to the composed modes (the all-to-all alone does not use it)
        const bool fused = mode == PERM_FUSED_FWD || mode == PERM_FUSED_INV;
        if (dk.bs != d[0].bs || dk.L != d[0].L || dk.rd != d[0].rd || dk.ud != d[0].ud ||
            (fused && dk.split != d[0].split))
            return USP_ERR_SHAPE;
        work += dk.bs * dk.L * (int64_t)dk.H;
        a.job[k] = PermJob{static_cast<const char *>(src[k]), static_cast<char *>(dst[k]), dk.H,
                           dk.H_total ? dk.H_total : dk.H, dk.h0, (int64_t)dk.hd * elem_size(dk.dtype), dk.dtype};
    }
    if (work == 0) return USP_OK;
    for (int k = 0; k < n; ++k) {
        if (d[k].H == 0) continue;
        if (!src[k] || !dst[k]) return USP_ERR_INVALID_ARG;
        int rc = check_ptr_align(src[k], dst[k], a.job[k].row_bytes);
        if (rc) return rc;
    }
    a.split = d[0].split;
    a.bs = d[0].bs; a.L = d[0].L;
    a.rd = d[0].rd; a.ud = d[0].ud;
    a.max_blocks = max_blocks;
    return launch_permute(a, reinterpret_cast<cudaStream_t>(stream));
}

int usp_extract_a2a(int n, const void *const *src, void *const *dst, const usp_dims *d, int inverse,
                    usp_stream_t stream) {
    return permute_multi(n, src, dst, d, inverse ? PERM_FUSED_INV : PERM_FUSED_FWD, stream);
}

int usp_a2a4d_multi(int n, const void *const *src, void *const *dst, const usp_dims *d, int dir,
                    usp_stream_t stream) {
    if (dir != 1 && dir != -1) return USP_ERR_INVALID_ARG;
    return permute_multi(n, src, dst, d, dir > 0 ? PERM_A2A_FWD : PERM_A2A_INV, stream);
}

// checks shared by the forward and backward attention entry points; fills the kernel arguments
static int check_attn_desc(const usp_attn_desc &d) {
    if (d.bs < 0 || d.L < 0 || d.hq <= 0 || d.hkv <= 0 || d.rd <= 0 || d.ud <= 0)
        return USP_ERR_INVALID_ARG;
    if (d.mode < USP_MODE_FUSED || d.mode > USP_MODE_ACCUM) return USP_ERR_INVALID_ARG;
    if (d.mode != USP_MODE_FUSED && (d.step < 0 || d.step >= d.rd)) return USP_ERR_INVALID_ARG;
    if (d.split < USP_SPLIT_ZIGZAG || d.split > USP_SPLIT_STRIPE) return USP_ERR_INVALID_ARG;
    if (d.ring_rank_only < 0 || d.ring_rank_only > d.rd) return USP_ERR_INVALID_ARG;
    if (elem_size(d.dtype) == 0) return USP_ERR_DTYPE;
    if (d.L % (2 * (int64_t)d.rd) != 0 || (d.L / d.rd) % d.ud != 0) return USP_ERR_SHAPE;
    if (d.hq % d.hkv != 0 || d.hq % d.ud != 0 || heads_per_rank(d.hkv, d.ud) == 0) return USP_ERR_SHAPE;
    if (d.hd != 64 && d.hd != 128) return USP_ERR_UNSUPPORTED;
    if (overflow31(d.bs * d.L * (int64_t)d.hq) || overflow31(d.L)) return USP_ERR_UNSUPPORTED;
    if (!(d.scale == d.scale) || isinf(d.scale)) return USP_ERR_INVALID_ARG;
    if (d.nseq < 0 || (d.nseq > 1 && (!d.cu_seqlens || !aligned(d.cu_seqlens, 4)))) return USP_ERR_INVALID_ARG;
    if (d.nseq > d.L) return USP_ERR_SHAPE;
    return USP_OK;
}

static AttnArgs attn_args(const usp_attn_desc &d) {
    AttnArgs a{};
    a.bs = d.bs; a.L = d.L; a.hq = d.hq; a.hkv = d.hkv; a.hd = d.hd; a.rd = d.rd; a.ud = d.ud;
    a.dtype = d.dtype; a.causal = d.causal ? 1 : 0; a.mode = d.mode; a.step = d.step;
    a.split = d.split; a.ring_rank_only = d.ring_rank_only;
    a.scale = d.scale > 0.f ? d.scale : 1.0f / sqrtf((float)d.hd);
    a.cu = d.nseq > 1 ? d.cu_seqlens : nullptr;
    a.nseq = d.nseq > 1 ? d.nseq : 0;
    return a;
}

int usp_attn_bwd_delta(const void *out, const void *dout, float *delta, int64_t rows, int32_t hd, int32_t dtype,
                       usp_stream_t stream) {
    if (rows < 0 || hd <= 0) return USP_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    if (es == 0) return USP_ERR_DTYPE;
    if (((int64_t)hd * es) % 16 != 0) return USP_ERR_UNSUPPORTED;
    if (overflow31(rows) || overflow31(rows * hd)) return USP_ERR_UNSUPPORTED;
    if (rows == 0) return USP_OK;
    if (!out || !dout || !delta) return USP_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(dout, 16) || !aligned(delta, 16)) return USP_ERR_ALIGN;
    return launch_row_dot(out, dout, delta, rows, hd, dtype, reinterpret_cast<cudaStream_t>(stream));
}

int usp_attn_bwd(const void *q, const void *k, const void *v, const void *dout, const float *lse, const float *delta,
                 void *dq, void *dk, void *dv, usp_attn_desc d, usp_stream_t stream) {
    int rc = check_attn_desc(d);
    if (rc) return rc;
    if (d.mode != USP_MODE_FUSED || d.ring_rank_only != 0) return USP_ERR_INVALID_ARG;
    if (d.bs == 0 || d.L == 0) return USP_OK;
    const void *ptrs[] = {q, k, v, dout, lse, delta, dq, dk, dv};
    for (const void *x : ptrs) {
        if (!x) return USP_ERR_INVALID_ARG;
        if (!aligned(x, 16)) return USP_ERR_ALIGN;
    }
    BwdArgs a{};
    a.f = attn_args(d);
    a.f.q = q; a.f.k = k; a.f.v = v;
    a.f.lse = const_cast<float *>(lse);
    a.dout = dout; a.delta = delta;
    a.dq = dq; a.dk = dk; a.dv = dv;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (d.dtype == USP_BF16) return launch_attn_bwd_tc(a, s);
    return launch_attn_bwd_simt(a, s);
}

int usp_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, usp_attn_desc d,
                 usp_stream_t stream) {
    return attn_fwd_capped(q, k, v, out, lse, d, 0, stream);
}

int usp_lse_merge(void *o_acc, float *lse_acc, const void *o_new, const float *lse_new, int64_t rows,
                  int32_t hd, int32_t dtype, usp_stream_t stream) {
    if (rows < 0 || hd <= 0) return USP_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    if (es == 0) return USP_ERR_DTYPE;
    if (((int64_t)hd * es) % 16 != 0) return USP_ERR_UNSUPPORTED;
    if (overflow31(rows) || overflow31(rows * hd)) return USP_ERR_UNSUPPORTED;
    if (rows == 0) return USP_OK;
    if (!o_acc || !lse_acc || !o_new || !lse_new) return USP_ERR_INVALID_ARG;
    if (!aligned(o_acc, 16) || !aligned(o_new, 16) || !aligned(lse_acc, 16) || !aligned(lse_new, 16))
        return USP_ERR_ALIGN;
    return launch_lse_merge(o_acc, lse_acc, o_new, lse_new, rows, hd, dtype,
                            reinterpret_cast<cudaStream_t>(stream));
}

int usp_selftest_timeout(int64_t limit_us, usp_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return USP_ERR_INVALID_ARG;
    const DeviceInfo *di = device_info();
    if (!di) return USP_ERR_CUDA;
    usp::selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(di->status,
                                                                                  (uint64_t)limit_us * 1000ull);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

int usp_check(usp_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return USP_ERR_CUDA;
    const DeviceInfo *di = device_info();
    if (!di) return USP_ERR_CUDA;
    int st = 0;
    if (cudaMemcpy(&st, di->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return USP_ERR_CUDA;
    if (st != 0) {
        int zero = 0;
        if (cudaMemcpy(di->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return USP_ERR_CUDA;
        return USP_ERR_TIMEOUT;
    }
    return USP_OK;
}

}  // extern "C"

namespace usp {

int extract_a2a_capped(int n, const void *const *src, void *const *dst, const usp_dims *d, int inverse,
                       int max_blocks, usp_stream_t stream) {
    return permute_multi(n, src, dst, d, inverse ? PERM_FUSED_INV : PERM_FUSED_FWD, stream, max_blocks);
}

int attn_fwd_capped(const void *q, const void *k, const void *v, void *out, float *lse, const usp_attn_desc &d,
                    int max_ctas, usp_stream_t stream) {
    int rc = check_attn_desc(d);
    if (rc) return rc;
    if (d.bs == 0 || d.L == 0) return USP_OK;
    if (!q || !k || !v || !out || !lse) return USP_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 16))
        return USP_ERR_ALIGN;
    AttnArgs a = attn_args(d);
    a.q = q; a.k = k; a.v = v; a.out = out; a.lse = lse;
    a.max_ctas = max_ctas;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (d.dtype == USP_BF16) {
        // the tensor-core launcher sets each kernel's shared-memory attribute on its first launch on
        // a device and remembers it; host threads launching at the same time take turns here
        static std::mutex tc_mu;
        std::lock_guard<std::mutex> lk(tc_mu);
        return launch_attn_tc(a, s);
    }
    return launch_attn_simt(a, s);
}

}  // namespace usp
