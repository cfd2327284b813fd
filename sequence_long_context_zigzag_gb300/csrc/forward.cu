// forward.cu -- the whole USP-Attention forward (steps a1-a5, plus the inverse split a7 back to
// natural order) as one call, on device buffers or pipelined from pinned host buffers; and the whole
// backward on device buffers.
//
// Per head group (UPipe-style head chunking): the composed zigzag split + AllToAll4D of Q, K, V, the
// fused ring attention, and the composed inverse of out and lse. The host-buffer variant overlaps,
// on three internal streams, the host-to-device copy of group g+1 and the device-to-host copy of
// group g-1 with the kernels of group g (two staging slots per direction) -- or, when the host
// buffers are mapped page-locked memory, lets the kernels read and write them directly.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// usp_forward_host's direct path runs a head group's host transfers beside the previous or next
// group's attention, on a few thread blocks each (a block holds at most one SM, which the persistent
// attention then leaves free). Blocks per transfer are chosen so that it moves its bytes in about
// half of the attention's time, from per-block rates over NVLink-C2C measured on GB300 (about 18 GB/s
// reading pinned host memory and 16 GB/s writing it; 210 and 159 GB/s uncapped) and the attention
// estimated at 1.5 PFLOP/s. More than kXferMaxBlocks per transfer: no overlap.
constexpr double kXferReadGBs = 18.0, kXferWriteGBs = 16.0, kXferAttnTflops = 1500.0;
constexpr int kXferMaxBlocks = 8;

struct FwdShape {
    int64_t bs, L;
    int hq, hkv, hd, rd, ud, hc, hkc, G, es, split;
    size_t q_grp, kv_grp, lse_grp;  // bytes of one group's q / k (or v) / lse, natural order
    size_t kv_hs;                   // bytes of one group's k (or v) head-sharded (more when replicated)
};

int fwd_shape(const usp_attn_desc &d, int head_chunk, FwdShape &s) {
    if (d.bs < 0 || d.L < 0 || d.hq <= 0 || d.hkv <= 0 || d.rd <= 0 || d.ud <= 0) return USP_ERR_INVALID_ARG;
    if (d.mode != USP_MODE_FUSED || d.ring_rank_only != 0) return USP_ERR_INVALID_ARG;
    s.es = elem_size(d.dtype);
    if (s.es == 0) return USP_ERR_DTYPE;
    if (d.hq % d.hkv != 0) return USP_ERR_SHAPE;
    s.bs = d.bs; s.L = d.L; s.hq = d.hq; s.hkv = d.hkv; s.hd = d.hd; s.rd = d.rd; s.ud = d.ud;
    s.G = d.hq / d.hkv;
    s.split = d.split;
    s.hc = head_chunk > 0 ? head_chunk : d.hq;
    if (s.hc > d.hq || d.hq % s.hc != 0 || s.hc % s.G != 0) return USP_ERR_SHAPE;
    s.hkc = s.hc / s.G;
    if (s.hc % d.ud != 0 || heads_per_rank(s.hkc, d.ud) == 0) return USP_ERR_SHAPE;
    const size_t tok = (size_t)d.bs * (size_t)d.L;
    s.q_grp = tok * s.hc * d.hd * s.es;
    s.kv_grp = tok * s.hkc * d.hd * s.es;
    s.kv_hs = tok * (size_t)heads_per_rank(s.hkc, d.ud) * d.ud * d.hd * s.es;
    s.lse_grp = tok * s.hc * 4;
    return USP_OK;
}

// workspace of the device-buffer forward: head-sharded q, k, v, out, lse of one group
size_t ws_device(const FwdShape &s) {
    return align_up(s.q_grp) * 2 + align_up(s.kv_hs) * 2 + align_up(s.lse_grp);
}

// workspace of the backward: D of all rows (natural), then per group head-sharded q, dout, dq,
// k, v, dk, dv, lse and D
size_t ws_backward(const FwdShape &s) {
    const size_t d_all = (size_t)s.bs * s.L * s.hq * 4;
    return align_up(d_all) + align_up(s.q_grp) * 3 + align_up(s.kv_hs) * 4 + align_up(s.lse_grp) * 2;
}

// the host-buffer forward: the copy path adds two slots of compact natural-order staging for q, k, v
// and out, and the full natural lse (copied back once at the end); the direct path takes two slots of
// the device buffers
size_t ws_host(const FwdShape &s) {
    const size_t lse_all = (size_t)s.bs * s.L * s.hq * 4;
    const size_t copy_path = ws_device(s) + 2 * (align_up(s.q_grp) * 2 + align_up(s.kv_grp) * 2) + align_up(lse_all);
    return std::max(copy_path, 2 * ws_device(s));  // the direct path: two slots of device buffers
}

struct Carve {
    char *p;
    size_t left;
    void *take(size_t n) {
        n = align_up(n);
        if (n > left) return nullptr;
        void *r = p;
        p += n;
        left -= n;
        return r;
    }
};

usp_dims dims_of(const FwdShape &s, int H, int H_total, int h0, int hd, int dtype) {
    usp_dims d{};
    d.bs = s.bs; d.L = s.L; d.H = H; d.hd = hd; d.dtype = dtype; d.rd = s.rd; d.ud = s.ud;
    d.H_total = H_total; d.h0 = h0; d.split = s.split;
    return d;
}

struct HostPipe {
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, in_ready[2] = {}, in_free[2] = {}, out_ready[2] = {}, out_free[2] = {},
                comp_done = nullptr, d2h_done = nullptr;
    bool ok = false;
};

constexpr int kMaxDev = 64;
HostPipe g_pipe[kMaxDev];
std::mutex g_pipe_mu[kMaxDev];

bool pipe_init(HostPipe &hp) {
    if (hp.ok) return true;
    const unsigned fl = cudaStreamNonBlocking;
    if (cudaStreamCreateWithFlags(&hp.h2d, fl) || cudaStreamCreateWithFlags(&hp.comp, fl) ||
        cudaStreamCreateWithFlags(&hp.d2h, fl))
        return false;
    cudaEvent_t *evs[] = {&hp.start, &hp.in_ready[0], &hp.in_ready[1], &hp.in_free[0], &hp.in_free[1],
                          &hp.out_ready[0], &hp.out_ready[1], &hp.out_free[0], &hp.out_free[1], &hp.comp_done,
                          &hp.d2h_done};
    for (cudaEvent_t *e : evs)
        if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
    hp.ok = true;
    return true;
}

struct XferPlan {
    int in_blocks = 0, out_blocks = 0;  // 0: the transfers do not run beside the attention
};

XferPlan xfer_plan(const FwdShape &s, const usp_attn_desc &d) {
    XferPlan x;
    // one group; packed samples (their cost is unknown here); fp32 (the attention is not persistent)
    if (s.hq / s.hc < 2 || d.nseq > 1 || d.dtype != USP_BF16) return x;
    const double flop = 4.0 * s.bs * s.hc * s.hd * (double)s.L * s.L * (d.causal ? 0.5 : 1.0);
    const double t_attn = flop / (kXferAttnTflops * 1e12);
    const double in_b = (double)s.bs * s.L * (s.hc + 2 * s.hkc) * s.hd * s.es;
    const double out_b = (double)s.bs * s.L * s.hc * ((double)s.hd * s.es + 4);
    const int bi = (int)std::ceil(2.0 * in_b / (kXferReadGBs * 1e9 * t_attn));
    const int bo = (int)std::ceil(2.0 * out_b / (kXferWriteGBs * 1e9 * t_attn));
    if (bi > kXferMaxBlocks || bo > kXferMaxBlocks) return x;
    x.in_blocks = std::max(bi, 1);
    x.out_blocks = std::max(bo, 1);
    return x;
}

// The forward of every head group on device buffers (usp_forward): the composed split + all-to-all
// of q, k, v, the ring attention, and the composed inverse of out and lse.
int forward_groups(const FwdShape &s, const usp_attn_desc &d, const void *q, const void *k, const void *v, void *out,
                   float *lse, void *qh, void *kh, void *vh, void *oh, float *lh, usp_stream_t stream) {
    int rc;
    for (int g0 = 0; g0 < s.hq; g0 += s.hc) {
        const int gk = g0 / s.G;
        const void *srcs[3] = {q, k, v};
        void *dsts[3] = {qh, kh, vh};
        usp_dims dd[3] = {dims_of(s, s.hc, s.hq, g0, s.hd, d.dtype), dims_of(s, s.hkc, s.hkv, gk, s.hd, d.dtype),
                          dims_of(s, s.hkc, s.hkv, gk, s.hd, d.dtype)};
        if ((rc = usp_extract_a2a(3, srcs, dsts, dd, 0, stream))) return rc;
        usp_attn_desc ad = d;
        ad.hq = s.hc;
        ad.hkv = s.hkc;
        if ((rc = usp_attn_fwd(qh, kh, vh, oh, lh, ad, stream))) return rc;
        // out and lse back to natural order in one launch
        const void *os[2] = {oh, lh};
        void *od[2] = {out, lse};
        usp_dims odims[2] = {dims_of(s, s.hc, s.hq, g0, s.hd, d.dtype), dims_of(s, s.hc, s.hq, g0, 1, USP_F32)};
        if ((rc = usp_extract_a2a(2, os, od, odims, 1, stream))) return rc;
    }
    return USP_OK;
}

// Device address of a host buffer that is page-locked and mapped into the current device's address
// space (cudaHostAlloc, cudaHostRegister, or a pinned torch tensor), else nullptr.
void *mapped_host(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer is not an error of the call; clear it
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// 2-D copy of a head window: `rows` rows of `width` bytes, source / destination pitches in bytes
inline bool copy2d(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, size_t rows,
                   cudaMemcpyKind kind, cudaStream_t s) {
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s) == cudaSuccess;
}

}  // namespace
}  // namespace usp

using namespace usp;

extern "C" {

size_t usp_forward_workspace_size(usp_attn_desc d, int head_chunk, int host_buffers) {
    FwdShape s{};
    if (fwd_shape(d, head_chunk, s) != USP_OK) return 0;
    return host_buffers ? ws_host(s) : ws_device(s);
}

int usp_forward(const void *q, const void *k, const void *v, void *out, float *lse, usp_attn_desc d, int head_chunk,
                void *workspace, size_t workspace_bytes, usp_stream_t stream) {
    FwdShape s{};
    int rc = fwd_shape(d, head_chunk, s);
    if (rc) return rc;
    if (d.bs == 0 || d.L == 0) return USP_OK;
    if (!q || !k || !v || !out || !lse || !workspace) return USP_ERR_INVALID_ARG;
    if (workspace_bytes < ws_device(s)) return USP_ERR_INVALID_ARG;
    if (!aligned(workspace, kAlign)) return USP_ERR_ALIGN;
    Carve cv{static_cast<char *>(workspace), workspace_bytes};
    void *qh = cv.take(s.q_grp), *kh = cv.take(s.kv_hs), *vh = cv.take(s.kv_hs), *oh = cv.take(s.q_grp);
    float *lh = static_cast<float *>(cv.take(s.lse_grp));
    return forward_groups(s, d, q, k, v, out, lse, qh, kh, vh, oh, lh, stream);
}

int usp_forward_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, float *lse_host,
                     usp_attn_desc d, int head_chunk, void *workspace, size_t workspace_bytes, usp_stream_t stream) {
    FwdShape s{};
    int rc = fwd_shape(d, head_chunk, s);
    if (rc) return rc;
    if (d.bs == 0 || d.L == 0) return USP_OK;
    if (!q_host || !k_host || !v_host || !out_host || !lse_host || !workspace) return USP_ERR_INVALID_ARG;
    if (workspace_bytes < ws_host(s)) return USP_ERR_INVALID_ARG;
    if (!aligned(workspace, kAlign)) return USP_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return USP_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_pipe_mu[dev]);
    HostPipe &hp = g_pipe[dev];
    if (!pipe_init(hp)) return USP_ERR_CUDA;
    cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);
    bool okc = true;
    auto chk = [&](bool c) { okc = okc && c; };
    // Direct path: when every host buffer is mapped page-locked memory, the kernels read q, k, v and
    // write out and lse in host memory themselves, over the CPU-GPU link (NVLink-C2C on GB300);
    // nothing is staged or copied by DMA. The head groups are pipelined over two slots of device
    // buffers: while group g's attention runs, group g + 1's split + all-to-all gathers its input from
    // host memory (one stream) and group g - 1's inverse scatters out and lse to host memory (another
    // stream). The persistent attention then leaves as many SMs as those two transfers have thread
    // blocks (xfer_plan); the first gather and the last scatter have the GPU to themselves and run
    // uncapped. Without a plan (xfer_plan: 0) every launch is uncapped and the transfers wait for
    // the SMs the attention holds.
    {
        void *qd = mapped_host(q_host), *kd = mapped_host(k_host), *vd = mapped_host(v_host);
        void *odh = mapped_host(out_host), *ldh = mapped_host(lse_host);
        if (qd && kd && vd && odh && ldh) {
            Carve cv{static_cast<char *>(workspace), workspace_bytes};
            void *qh[2], *kh[2], *vh[2], *oh[2];
            float *lh[2];
            for (int b = 0; b < 2; ++b) {
                qh[b] = cv.take(s.q_grp);
                kh[b] = cv.take(s.kv_hs);
                vh[b] = cv.take(s.kv_hs);
                oh[b] = cv.take(s.q_grp);
                lh[b] = static_cast<float *>(cv.take(s.lse_grp));
            }
            if (!lh[1]) return USP_ERR_INVALID_ARG;
            const int ngroups = s.hq / s.hc;
            const XferPlan xp = xfer_plan(s, d);
            const DeviceInfo *di = device_info();
            if (!di) return USP_ERR_CUDA;
            const int attn_ctas = xp.in_blocks ? std::max(1, di->sm_count - xp.in_blocks - xp.out_blocks) : 0;
            usp_stream_t gat = reinterpret_cast<usp_stream_t>(hp.h2d), sca = reinterpret_cast<usp_stream_t>(hp.d2h);
            auto gather = [&](int g, usp_stream_t st, int max_blocks) {
                const int g0 = g * s.hc, gk = g0 / s.G, b = g & 1;
                const void *srcs[3] = {qd, kd, vd};
                void *dsts[3] = {qh[b], kh[b], vh[b]};
                usp_dims dd[3] = {dims_of(s, s.hc, s.hq, g0, s.hd, d.dtype),
                                  dims_of(s, s.hkc, s.hkv, gk, s.hd, d.dtype),
                                  dims_of(s, s.hkc, s.hkv, gk, s.hd, d.dtype)};
                return extract_a2a_capped(3, srcs, dsts, dd, 0, max_blocks, st);
            };
            auto scatter = [&](int g, usp_stream_t st, int max_blocks) {
                const int g0 = g * s.hc, b = g & 1;
                const void *os[2] = {oh[b], lh[b]};
                void *od[2] = {odh, ldh};
                usp_dims odims[2] = {dims_of(s, s.hc, s.hq, g0, s.hd, d.dtype),
                                     dims_of(s, s.hc, s.hq, g0, 1, USP_F32)};
                return extract_a2a_capped(2, os, od, odims, 1, max_blocks, st);
            };
            // an error after work was queued still orders the caller's stream after everything this
            // call put on the library's streams
            auto fail = [&](int code) {
                cudaEventRecord(hp.comp_done, hp.h2d);
                cudaStreamWaitEvent(user, hp.comp_done, 0);
                cudaEventRecord(hp.d2h_done, hp.d2h);
                cudaStreamWaitEvent(user, hp.d2h_done, 0);
                return code;
            };
            chk(cudaEventRecord(hp.start, user) == cudaSuccess);
            chk(cudaStreamWaitEvent(hp.h2d, hp.start, 0) == cudaSuccess);
            chk(cudaStreamWaitEvent(hp.d2h, hp.start, 0) == cudaSuccess);
            if ((rc = gather(0, stream, 0))) return fail(rc);
            for (int g = 0; g < ngroups && okc; ++g) {
                const int b = g & 1;
                // inputs of slot b gathered (group 0: earlier on this stream); outputs of slot b
                // scattered (group g - 2)
                if (g > 0) chk(cudaStreamWaitEvent(user, hp.in_ready[b], 0) == cudaSuccess);
                if (g > 1) chk(cudaStreamWaitEvent(user, hp.out_free[b], 0) == cudaSuccess);
                usp_attn_desc ad = d;
                ad.hq = s.hc;
                ad.hkv = s.hkc;
                if ((rc = attn_fwd_capped(qh[b], kh[b], vh[b], oh[b], lh[b], ad, attn_ctas, stream))) return fail(rc);
                chk(cudaEventRecord(hp.in_free[b], user) == cudaSuccess);  // slot b's inputs read, outputs written
                if (g + 1 < ngroups) {
                    // group g + 1 into the other slot, once group g - 1's attention has read it
                    if (g > 0) chk(cudaStreamWaitEvent(hp.h2d, hp.in_free[b ^ 1], 0) == cudaSuccess);
                    if ((rc = gather(g + 1, gat, xp.in_blocks))) return fail(rc);
                    chk(cudaEventRecord(hp.in_ready[b ^ 1], hp.h2d) == cudaSuccess);
                }
                chk(cudaStreamWaitEvent(hp.d2h, hp.in_free[b], 0) == cudaSuccess);
                if ((rc = scatter(g, sca, g + 1 < ngroups ? xp.out_blocks : 0))) return fail(rc);
                chk(cudaEventRecord(hp.out_free[b], hp.d2h) == cudaSuccess);
            }
            chk(cudaEventRecord(hp.d2h_done, hp.d2h) == cudaSuccess);
            chk(cudaStreamWaitEvent(user, hp.d2h_done, 0) == cudaSuccess);
            return okc ? USP_OK : USP_ERR_CUDA;
        }
    }
    // Copy path (pageable or unmapped host buffers): staged DMA copies of each head group's window,
    // pipelined with the kernels on the library's streams.

    Carve cv{static_cast<char *>(workspace), workspace_bytes};
    void *qh = cv.take(s.q_grp), *kh = cv.take(s.kv_hs), *vh = cv.take(s.kv_hs), *oh = cv.take(s.q_grp);
    float *lh = static_cast<float *>(cv.take(s.lse_grp));
    void *in_q[2], *in_k[2], *in_v[2], *out_o[2];
    for (int sl = 0; sl < 2; ++sl) {
        in_q[sl] = cv.take(s.q_grp);
        in_k[sl] = cv.take(s.kv_grp);
        in_v[sl] = cv.take(s.kv_grp);
        out_o[sl] = cv.take(s.q_grp);
    }
    float *lse_all = static_cast<float *>(cv.take((size_t)s.bs * s.L * s.hq * 4));
    if (!lse_all) return USP_ERR_INVALID_ARG;

    const size_t rows = (size_t)s.bs * s.L;
    const size_t row_q = (size_t)s.hd * s.es;  // bytes of one (token, head) row
    auto fail = [&](int code) {  // as in the direct path: the caller's stream after all queued work
        cudaEventRecord(hp.in_ready[0], hp.h2d);
        cudaStreamWaitEvent(user, hp.in_ready[0], 0);
        cudaEventRecord(hp.comp_done, hp.comp);
        cudaStreamWaitEvent(user, hp.comp_done, 0);
        cudaEventRecord(hp.d2h_done, hp.d2h);
        cudaStreamWaitEvent(user, hp.d2h_done, 0);
        return code;
    };
    chk(cudaEventRecord(hp.start, user) == cudaSuccess);
    chk(cudaStreamWaitEvent(hp.h2d, hp.start, 0) == cudaSuccess);
    chk(cudaStreamWaitEvent(hp.comp, hp.start, 0) == cudaSuccess);
    chk(cudaStreamWaitEvent(hp.d2h, hp.start, 0) == cudaSuccess);
    const int ngroups = s.hq / s.hc;
    for (int g = 0; g < ngroups && okc; ++g) {
        const int sl = g & 1;
        const int g0 = g * s.hc, gk = g0 / s.G;
        // host -> device: this group's head windows into compact natural-order staging
        if (g >= 2) chk(cudaStreamWaitEvent(hp.h2d, hp.in_free[sl], 0) == cudaSuccess);
        chk(copy2d(in_q[sl], s.hc * row_q, static_cast<const char *>(q_host) + g0 * row_q, s.hq * row_q,
                   s.hc * row_q, rows, cudaMemcpyHostToDevice, hp.h2d));
        chk(copy2d(in_k[sl], s.hkc * row_q, static_cast<const char *>(k_host) + gk * row_q, s.hkv * row_q,
                   s.hkc * row_q, rows, cudaMemcpyHostToDevice, hp.h2d));
        chk(copy2d(in_v[sl], s.hkc * row_q, static_cast<const char *>(v_host) + gk * row_q, s.hkv * row_q,
                   s.hkc * row_q, rows, cudaMemcpyHostToDevice, hp.h2d));
        chk(cudaEventRecord(hp.in_ready[sl], hp.h2d) == cudaSuccess);
        // kernels
        usp_stream_t cs = reinterpret_cast<usp_stream_t>(hp.comp);
        chk(cudaStreamWaitEvent(hp.comp, hp.in_ready[sl], 0) == cudaSuccess);
        const void *srcs[3] = {in_q[sl], in_k[sl], in_v[sl]};
        void *dsts[3] = {qh, kh, vh};
        usp_dims dd[3] = {dims_of(s, s.hc, s.hc, 0, s.hd, d.dtype), dims_of(s, s.hkc, s.hkc, 0, s.hd, d.dtype),
                          dims_of(s, s.hkc, s.hkc, 0, s.hd, d.dtype)};
        if ((rc = usp_extract_a2a(3, srcs, dsts, dd, 0, cs))) return fail(rc);
        chk(cudaEventRecord(hp.in_free[sl], hp.comp) == cudaSuccess);
        usp_attn_desc ad = d;
        ad.hq = s.hc;
        ad.hkv = s.hkc;
        if ((rc = usp_attn_fwd(qh, kh, vh, oh, lh, ad, cs))) return fail(rc);
        if (g >= 2) chk(cudaStreamWaitEvent(hp.comp, hp.out_free[sl], 0) == cudaSuccess);
        const void *os[2] = {oh, lh};
        void *od[2] = {out_o[sl], lse_all};
        usp_dims odims[2] = {dims_of(s, s.hc, s.hc, 0, s.hd, d.dtype), dims_of(s, s.hc, s.hq, g0, 1, USP_F32)};
        if ((rc = usp_extract_a2a(2, os, od, odims, 1, cs))) return fail(rc);
        chk(cudaEventRecord(hp.out_ready[sl], hp.comp) == cudaSuccess);
        // device -> host: this group's output window
        chk(cudaStreamWaitEvent(hp.d2h, hp.out_ready[sl], 0) == cudaSuccess);
        chk(copy2d(static_cast<char *>(out_host) + g0 * row_q, s.hq * row_q, out_o[sl], s.hc * row_q, s.hc * row_q,
                   rows, cudaMemcpyDeviceToHost, hp.d2h));
        chk(cudaEventRecord(hp.out_free[sl], hp.d2h) == cudaSuccess);
    }
    // lse (small) in one copy once every group has written its window
    chk(cudaEventRecord(hp.comp_done, hp.comp) == cudaSuccess);
    chk(cudaStreamWaitEvent(hp.d2h, hp.comp_done, 0) == cudaSuccess);
    chk(cudaMemcpyAsync(lse_host, lse_all, (size_t)s.bs * s.L * s.hq * 4, cudaMemcpyDeviceToHost, hp.d2h) ==
        cudaSuccess);
    chk(cudaEventRecord(hp.d2h_done, hp.d2h) == cudaSuccess);
    chk(cudaStreamWaitEvent(user, hp.d2h_done, 0) == cudaSuccess);
    return okc ? USP_OK : USP_ERR_CUDA;
}

size_t usp_backward_workspace_size(usp_attn_desc d, int head_chunk) {
    FwdShape s{};
    if (fwd_shape(d, head_chunk, s) != USP_OK) return 0;
    return ws_backward(s);
}

int usp_backward(const void *q, const void *k, const void *v, const void *out, const float *lse, const void *dout,
                 void *dq, void *dk, void *dv, usp_attn_desc d, int head_chunk, void *workspace,
                 size_t workspace_bytes, usp_stream_t stream) {
    FwdShape s{};
    int rc = fwd_shape(d, head_chunk, s);
    if (rc) return rc;
    if (d.bs == 0 || d.L == 0) return USP_OK;
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !workspace) return USP_ERR_INVALID_ARG;
    if (workspace_bytes < ws_backward(s)) return USP_ERR_INVALID_ARG;
    if (!aligned(workspace, kAlign)) return USP_ERR_ALIGN;
    Carve cv{static_cast<char *>(workspace), workspace_bytes};
    float *d_all = static_cast<float *>(cv.take((size_t)s.bs * s.L * s.hq * 4));
    void *qh = cv.take(s.q_grp), *gh = cv.take(s.q_grp), *dqh = cv.take(s.q_grp);
    void *kh = cv.take(s.kv_hs), *vh = cv.take(s.kv_hs), *dkh = cv.take(s.kv_hs), *dvh = cv.take(s.kv_hs);
    float *lh = static_cast<float *>(cv.take(s.lse_grp)), *dh = static_cast<float *>(cv.take(s.lse_grp));
    // D = <dout, out> for every (token, query head), natural layout
    if ((rc = usp_attn_bwd_delta(out, dout, d_all, s.bs * s.L * s.hq, s.hd, d.dtype, stream))) return rc;
    for (int g0 = 0; g0 < s.hq; g0 += s.hc) {
        const int gk = g0 / s.G;
        const void *srcs[4] = {q, k, v, dout};
        void *dsts[4] = {qh, kh, vh, gh};
        usp_dims dd[4] = {dims_of(s, s.hc, s.hq, g0, s.hd, d.dtype), dims_of(s, s.hkc, s.hkv, gk, s.hd, d.dtype),
                          dims_of(s, s.hkc, s.hkv, gk, s.hd, d.dtype), dims_of(s, s.hc, s.hq, g0, s.hd, d.dtype)};
        if ((rc = usp_extract_a2a(4, srcs, dsts, dd, 0, stream))) return rc;
        const void *ls[2] = {lse, d_all};
        void *ld[2] = {lh, dh};
        usp_dims ldims[2] = {dims_of(s, s.hc, s.hq, g0, 1, USP_F32), dims_of(s, s.hc, s.hq, g0, 1, USP_F32)};
        if ((rc = usp_extract_a2a(2, ls, ld, ldims, 0, stream))) return rc;
        usp_attn_desc ad = d;
        ad.hq = s.hc;
        ad.hkv = s.hkc;
        if ((rc = usp_attn_bwd(qh, kh, vh, gh, lh, dh, dqh, dkh, dvh, ad, stream))) return rc;
        // the gradients back to natural order in one call: inverse all-to-all and split (the KV
        // gradients of replicated heads sum their replicas, in a launch of their own)
        const void *gs[3] = {dqh, dkh, dvh};
        void *gd[3] = {dq, dk, dv};
        usp_dims gdims[3] = {dims_of(s, s.hc, s.hq, g0, s.hd, d.dtype), dims_of(s, s.hkc, s.hkv, gk, s.hd, d.dtype),
                             dims_of(s, s.hkc, s.hkv, gk, s.hd, d.dtype)};
        if ((rc = usp_extract_a2a(3, gs, gd, gdims, 1, stream))) return rc;
    }
    return USP_OK;
}

}  // extern "C"
