// attn_bwd_tc.cu -- bf16 ring attention backward on the 5th-generation tensor cores (sm_103a).
//
// What it computes: the gradients of the forward (chain rule through softmax), over the forward's
// causal (query, key) pairs of the ring (every ring rank's queries meet every rank's KV block once):
//   P_ij = exp(s_ij - lse_i),  dP_ij = <dout_i, v_j>,  dS_ij = P_ij (dP_ij - D_i),  D_i = <dout_i, out_i>
//   dv_j = sum_i P_ij dout_i,  dk_j = scale sum_i dS_ij q_i,  dq_i = scale sum_j dS_ij k_j.
// In a multi-GPU ring the dk/dv partials would travel with their KV block and be home after rd steps
// (the Context-Parallel page pairs the forward's KV gather with a reduce-scatter of the gradients);
// here each kernel forms a whole gradient tile on one SM, so nothing is exchanged or accumulated in
// global memory (no atomics, deterministic).
//
// Two kernels, each with the same warp layout (384 threads):
//   warps 0-3 and 4-7   "softmax": one thread per TMEM lane (a row of the CTA's tile); warpgroup w
//                       handles columns [32 w, 32 w + 32) of each 64-column score tile;
//   warp 8              TMA producer (whole warp: lane 0 issues copies, all lanes stage lse / D);
//   warp 9              allocates tensor memory; lane 0 issues every MMA and commit.
// dk/dv kernel (CTA = 128 keys of one (ring rank s, Ulysses rank u, KV head, batch)): K and V stay in
// shared memory; 64-row tiles of Q and dout (and their lse, D) stream through a ring of stages, for
// every ring rank's queries that see the keys and every query head of the KV head's group. Per Q tile
// t (TMEM buffer b = t mod 2):
//   S^T_b = K Q_t^T, dP^T_b = V dout_t^T          (M = 128 keys, N = 64 queries, K = hd; from smem)
//   softmax: P^T = exp2(S^T scale log2e - lse log2e) (0 where masked), dS^T = P^T (dP^T - D), both
//            bf16, written back over the first 16 columns of each warpgroup's half
//   dV += P^T dout_t, dK += dS^T Q_t               (M = 128 keys, N = hd, K = 64; A from TMEM, B
//                                                   = dout_t / Q_t viewed MN-major)
// issued as SP(t+2) right after ACC(t), so the softmax of tile t+1 runs while the tensor core works
// on tiles t and t+2.
// dq kernel (CTA = 128 queries of one (r, u, query head, batch)): Q and dout stay; 64-key tiles of K
// and V stream over the ring steps in the Context-Parallel page's Fig. 1 order, visible prefixes only:
//   S_b = Q K_t^T, dP_b = dout V_t^T,  dS_b = P (dP - D),  dQ += dS_b K_t.
// TMEM (512 columns): dk/dv kernel: dV [0,hd) dK [hd,2hd) S^T_b 2hd + 128b + [0,64) dP^T_b + [64,128);
// dq kernel: dQ [0,hd) S_b hd + 128b + [0,64) dP_b + [64,128).
// Every wait is bounded (2 s): on expiry the kernel records USP_ERR_TIMEOUT, drains and returns.
#include <cuda.h>
#include <mutex>

#include "tc_common.cuh"
#include "tc_ptx.cuh"
#include "usp_device.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kT = 64;  // rows of a streamed tile (queries in the dk/dv kernel, keys in the dq kernel)
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdTcParams {
    CUtensorMap t_big0, t_big1;      // 128-row boxes: K, V (dk/dv kernel) or Q, dout (dq kernel)
    CUtensorMap t_small0, t_small1;  // 64-row boxes: Q, dout (dk/dv kernel) or K, V (dq kernel)
    const float *lse, *delta;
    __nv_bfloat16 *g0, *g1;          // dk, dv (dk/dv kernel) or dq (dq kernel)
    int *status;
    uint32_t bs, Lr, c, rd, ud, Hl, Hkl, G, ntiles;  // ntiles: 128-row tiles per ring-local block
    int causal, split, lpt;
    float scale, scale_log2;
    const int32_t *cu;  // packed samples' cumulative lengths, or nullptr
    uint32_t nseq, L;
};

template <int HD> struct Lay {
    static constexpr int kBoxes = HD / 64;
    static constexpr int kBigBox = 128 * 128;   // 128 rows x 128 bytes
    static constexpr int kBigTile = 128 * HD * 2;
    static constexpr int kSmallBox = kT * 128;  // 64 rows x 128 bytes
    static constexpr int kSmallTile = kT * HD * 2;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// S(^T) and dP(^T) of one tile: D_s = A0 B0^T, D_p = A1 B1^T with 128-row A tiles and 64-row B tiles,
// both K-major in 128-byte-swizzled boxes (M = 128, N = 64, K = hd)
template <int HD>
__device__ __forceinline__ void issue_sp(uint32_t t_s, uint32_t t_p, uint64_t a0, uint64_t b0, uint64_t a1,
                                         uint64_t b1) {
    using Y = Lay<HD>;
    constexpr uint32_t id = tc::idesc_bf16_f32(128, kT, 0, 0);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint64_t ao = (uint64_t)(((kk / 4) * Y::kBigBox + (kk % 4) * 32) >> 4);
        const uint64_t bo = (uint64_t)(((kk / 4) * Y::kSmallBox + (kk % 4) * 32) >> 4);
        tc::mma_ss(t_s, a0 + ao, b0 + bo, id, kk > 0 ? 1u : 0u);
    }
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint64_t ao = (uint64_t)(((kk / 4) * Y::kBigBox + (kk % 4) * 32) >> 4);
        const uint64_t bo = (uint64_t)(((kk / 4) * Y::kSmallBox + (kk % 4) * 32) >> 4);
        tc::mma_ss(t_p, a1 + ao, b1 + bo, id, kk > 0 ? 1u : 0u);
    }
}

// D (+)= A[tmem] B: A is a 128 x 64 bf16 tile held in TMEM as two 32-column halves, each packed into
// the first 16 columns of its 32-column half (k-step kk: column 32 (kk / 2) + 8 (kk % 2)); B is a
// 64-row tile viewed MN-major (N = hd: 64-column blocks kSmallBox apart, 8-row groups 1024 apart)
template <int HD>
__device__ __forceinline__ void issue_acc(uint32_t t_d, uint32_t t_a, uint64_t bdesc, uint32_t accumulate) {
    constexpr uint32_t id = tc::idesc_bf16_f32(128, HD, 0, 1);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk)
        tc::mma_ts(t_d, t_a + 32u * (kk / 2) + 8u * (kk % 2), bdesc + (uint64_t)((kk * 2048) >> 4), id,
                   (accumulate || kk > 0) ? 1u : 0u);
}

// one 32-column half of a score tile: P = exp2(s * sl2 - lse2) where visible (0 elsewhere),
// dS = P (dP - D); lse2 / D are per column (dk/dv kernel) or per row (dq kernel, broadcast)
__device__ __forceinline__ void p_ds_half(const uint32_t (&sv)[32], const uint32_t (&dpv)[32], const float *lse2,
                                          const float *dd, float sl2, int lo, int hi, uint32_t (&pk)[16],
                                          uint32_t (&dk)[16]) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const bool v0 = e >= lo && e < hi, v1 = e + 1 >= lo && e + 1 < hi;
        const float p0 = v0 ? tc::ex2(fmaf(u2f(sv[e]), sl2, -lse2[e])) : 0.f;
        const float p1 = v1 ? tc::ex2(fmaf(u2f(sv[e + 1]), sl2, -lse2[e + 1])) : 0.f;
        const float d0 = p0 * (u2f(dpv[e]) - dd[e]);
        const float d1 = p1 * (u2f(dpv[e + 1]) - dd[e + 1]);
        pk[e / 2] = float2_to_bf16x2(p0, p1);
        dk[e / 2] = float2_to_bf16x2(d0, d1);
    }
}

// write a 128 x (32 columns) fp32 accumulator chunk of one thread's row as bf16
__device__ __forceinline__ void store_row32(__nv_bfloat16 *dst, const uint32_t (&o)[32], float mul) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = float2_to_bf16x2(u2f(o[q * 8 + 0]) * mul, u2f(o[q * 8 + 1]) * mul);
        w.y = float2_to_bf16x2(u2f(o[q * 8 + 2]) * mul, u2f(o[q * 8 + 3]) * mul);
        w.z = float2_to_bf16x2(u2f(o[q * 8 + 4]) * mul, u2f(o[q * 8 + 5]) * mul);
        w.w = float2_to_bf16x2(u2f(o[q * 8 + 6]) * mul, u2f(o[q * 8 + 7]) * mul);
        d[q] = w;
    }
}

__device__ __forceinline__ void store_zero32(__nv_bfloat16 *dst) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) d[q] = make_uint4(0, 0, 0, 0);
}

// ================================================================================================
// dk / dv kernel
// ================================================================================================
template <int HD> struct KvCfg : Lay<HD> {
    using Y = Lay<HD>;
    static constexpr int kStages = HD == 128 ? 4 : 6;
    static constexpr int kK = 0;
    static constexpr int kV = Y::kBigTile;
    static constexpr int kQ = 2 * Y::kBigTile;              // stage s: Q at kQ + s * kStage, dout + kSmallTile
    static constexpr int kStage = 2 * Y::kSmallTile;
    static constexpr int kVec = kQ + kStages * kStage;     // lse2[stages][64], then D[stages][64]
    static constexpr int kBar = kVec + kStages * 2 * kT * 4;
    static constexpr int KV_FULL = 0;
    static constexpr int QD_FULL = 1;                       // [stages], 32 arrivals (producer lanes)
    static constexpr int QD_EMPTY = QD_FULL + kStages;      // [stages]
    static constexpr int SP_FULL = QD_EMPTY + kStages;      // [2]
    static constexpr int P_FULL = SP_FULL + 2;              // [2], 8 arrivals (softmax warps)
    static constexpr int ACC_FULL = P_FULL + 2;
    static constexpr int DONE = ACC_FULL + 1;
    static constexpr int kNumBars = DONE + 1;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kSmemBytes = kTmemSlot + 16 + 1024;
    __device__ static constexpr uint32_t colS(int b) { return 2u * HD + 128u * (uint32_t)b; }
    __device__ static constexpr uint32_t colP(int b) { return 2u * HD + 128u * (uint32_t)b + 64u; }
};

struct KvWork {
    uint32_t s, u, kh, b, k0;
    uint32_t kv_row0;            // row of local key 0 of (s, u, kh, b) in k / v / dk / dv
    uint32_t kpos_min, kpos_max;
    uint32_t hbeg, hend;         // the rank's query heads that read this KV head
    uint32_t sa_first, se_last;  // sample start of the first key, sample end of the last (packed)
};

__device__ __forceinline__ KvWork kv_decode(const BwdTcParams &p) {
    KvWork w;
    const uint32_t inner = p.ud * p.Hkl * p.bs;
    const uint32_t outer = blockIdx.x / inner;
    uint32_t in = blockIdx.x % inner;
    w.kh = in % p.Hkl;
    in /= p.Hkl;
    w.b = in % p.bs;
    w.u = in / p.bs;
    if (p.lpt) {
        // zigzag with whole 128-row blocks per chunk: earliest positions (seen by most queries) first
        const uint32_t per_chunk = p.c / 128;
        const uint32_t a = outer / per_chunk, off = (outer % per_chunk) * 128;
        w.s = a < p.rd ? a : 2 * p.rd - 1 - a;
        w.k0 = (a < p.rd ? 0 : p.c) + off;
    } else if (p.split == USP_SPLIT_BASIC) {
        w.s = outer / p.ntiles;
        w.k0 = (outer % p.ntiles) * 128;
    } else {
        w.s = outer % p.rd;
        w.k0 = (outer / p.rd) * 128;
    }
    w.kv_row0 = (((w.s * p.ud + w.u) * p.Hkl + w.kh) * p.bs + w.b) * p.Lr;
    w.kpos_min = pos32(p.split, w.s, w.k0, p.c, p.rd);
    w.kpos_max = pos32(p.split, w.s, min(w.k0 + 127, p.Lr - 1), p.c, p.rd);
    w.hbeg = w.kh * p.G;
    w.hend = min(w.hbeg + p.G, p.Hl);
    w.sa_first = 0;
    w.se_last = p.L;
    if (p.cu) {
        uint32_t a, e;
        sample_bounds(p.cu, p.nseq, w.kpos_min, p.L, w.sa_first, e);
        sample_bounds(p.cu, p.nseq, w.kpos_max, p.L, a, w.se_last);
    }
    return w;
}

// the Q tiles that see the CTA's keys: ring ranks r, query heads h of the group, 64-row tiles n over
// the rows of rank r that see at least one of the keys -- from the first row that sees the earliest
// key (the first row of its sample without the causal mask) to the end of the last key's sample
// (the end of the block unless samples are packed)
struct QIter {
    uint32_t r, h, n, nlo, nhi;
    bool done;
};

__device__ __forceinline__ void kv_query_range(const BwdTcParams &p, const KvWork &w, uint32_t r, uint32_t &nlo,
                                               uint32_t &nhi) {
    const uint32_t ilo = before32(p.split, p.causal ? w.kpos_min : w.sa_first, r, p.c, p.rd);
    const uint32_t ihi = before32(p.split, w.se_last, r, p.c, p.rd);
    nlo = ilo / kT;
    nhi = ihi > ilo ? (ihi + kT - 1) / kT : nlo;
}

__device__ __forceinline__ void qiter_rank(const BwdTcParams &p, const KvWork &w, QIter &it) {
    kv_query_range(p, w, it.r, it.nlo, it.nhi);
    it.h = w.hbeg;
    it.n = it.nlo;
}

__device__ __forceinline__ void qiter_init(const BwdTcParams &p, const KvWork &w, QIter &it) {
    it.r = 0;
    it.done = false;
    qiter_rank(p, w, it);
    while (!it.done && (it.nlo >= it.nhi || w.hbeg >= w.hend)) {
        if (++it.r >= p.rd) it.done = true;
        else qiter_rank(p, w, it);
    }
}

__device__ __forceinline__ void qiter_advance(const BwdTcParams &p, const KvWork &w, QIter &it) {
    if (++it.n < it.nhi) return;
    it.n = it.nlo;
    if (++it.h < w.hend) return;
    do {
        if (++it.r >= p.rd) {
            it.done = true;
            return;
        }
        qiter_rank(p, w, it);
    } while (it.nlo >= it.nhi);
}

__device__ __forceinline__ uint32_t kv_count_tiles(const BwdTcParams &p, const KvWork &w) {
    uint32_t n = 0;
    for (uint32_t r = 0; r < p.rd; ++r) {
        uint32_t nlo, nhi;
        kv_query_range(p, w, r, nlo, nhi);
        if (nhi > nlo) n += (nhi - nlo) * (w.hend - w.hbeg);
    }
    return n;
}

template <int HD>
__device__ void kv_producer(const BwdTcParams &p, const KvWork &w, uint32_t sbase, uint32_t bar0, float *vec) {
    using C = KvCfg<HD>;
    const int lane = threadIdx.x & 31;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    auto wait = [&](int bar, uint32_t parity) {
        return tc::mbar_wait(BAR(bar), parity, p.status, USP_ERR_TIMEOUT, kWaitNs);
    };
    if (lane == 0) {
        tc::mbar_arrive_expect_tx(BAR(C::KV_FULL), 2 * C::kBigTile);
        for (int bx = 0; bx < C::kBoxes; ++bx) {
            tc::tma_load_2d(sbase + C::kK + bx * C::kBigBox, &p.t_big0, bx * 64, (int32_t)(w.kv_row0 + w.k0),
                            BAR(C::KV_FULL));
            tc::tma_load_2d(sbase + C::kV + bx * C::kBigBox, &p.t_big1, bx * 64, (int32_t)(w.kv_row0 + w.k0),
                            BAR(C::KV_FULL));
        }
    }
    QIter it;
    qiter_init(p, w, it);
    uint32_t t = 0;
    bool ok = true;
    while (!it.done) {
        const uint32_t st = t % C::kStages;
        ok = wait(C::QD_EMPTY + st, ((t / C::kStages) & 1u) ^ 1u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t q_row = (((it.r * p.ud + w.u) * p.Hl + it.h) * p.bs + w.b) * p.Lr + it.n * kT;
        float *l2 = vec + st * kT, *dd = vec + C::kStages * kT + st * kT;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t cidx = lane + 32 * k;
            const bool in = it.n * kT + cidx < p.Lr;
            l2[cidx] = in ? p.lse[q_row + cidx] * kLog2e : 0.f;
            dd[cidx] = in ? p.delta[q_row + cidx] : 0.f;
        }
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(BAR(C::QD_FULL + st), 2 * C::kSmallTile);
            const uint32_t sq = sbase + C::kQ + st * C::kStage;
            for (int bx = 0; bx < C::kBoxes; ++bx) {
                tc::tma_load_2d(sq + bx * C::kSmallBox, &p.t_small0, bx * 64, (int32_t)q_row, BAR(C::QD_FULL + st));
                tc::tma_load_2d(sq + C::kSmallTile + bx * C::kSmallBox, &p.t_small1, bx * 64, (int32_t)q_row,
                                BAR(C::QD_FULL + st));
            }
        } else {
            tc::mbar_arrive(BAR(C::QD_FULL + st));
        }
        ++t;
        qiter_advance(p, w, it);
    }
    if (!ok && lane == 0) {
        // drain the copies this warp issued before the CTA exits
        wait(C::KV_FULL, 0);
        for (uint32_t f = t > C::kStages ? t - C::kStages : 0; f < t; ++f)
            wait(C::QD_FULL + f % C::kStages, (f / C::kStages) & 1u);
    }
}

template <int HD>
__device__ void kv_mma(const BwdTcParams &p, const KvWork &w, uint32_t sbase, uint32_t bar0, uint32_t tmem) {
    using C = KvCfg<HD>;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    auto wait = [&](int bar, uint32_t parity) {
        return tc::mbar_wait(BAR(bar), parity, p.status, USP_ERR_TIMEOUT, kWaitNs);
    };
    const uint32_t n = kv_count_tiles(p, w);
    const uint64_t kdesc = tc::sw128_desc(sbase + C::kK, 16, 1024);
    const uint64_t vdesc = tc::sw128_desc(sbase + C::kV, 16, 1024);
    const uint64_t qk0 = tc::sw128_desc(sbase + C::kQ, 16, 1024);                           // K-major view
    const uint64_t qm0 = tc::sw128_desc(sbase + C::kQ, C::kSmallBox, 1024);                 // MN-major view
    auto soff = [](uint32_t st) { return (uint64_t)((st * C::kStage) >> 4); };
    constexpr uint64_t kDo = (uint64_t)(C::kSmallTile >> 4);
    auto sp = [&](uint32_t t) {
        const uint32_t st = t % C::kStages, b = t & 1u;
        if (!wait(C::QD_FULL + st, (t / C::kStages) & 1u)) return false;
        issue_sp<HD>(tmem + C::colS(b), tmem + C::colP(b), kdesc, qk0 + soff(st), vdesc, qk0 + soff(st) + kDo);
        tc::mma_commit(BAR(C::SP_FULL + b));
        return true;
    };
    bool ok = wait(C::KV_FULL, 0);
    if (ok && n > 0) ok = sp(0);
    if (ok && n > 1) ok = sp(1);
    for (uint32_t t = 0; ok && t < n; ++t) {
        const uint32_t st = t % C::kStages, b = t & 1u;
        if (!(ok = wait(C::P_FULL + b, (t >> 1) & 1u))) break;
        tc::fence_after_sync();
        issue_acc<HD>(tmem + 0, tmem + C::colS(b), qm0 + soff(st) + kDo, t > 0);  // dV += P^T dout
        issue_acc<HD>(tmem + HD, tmem + C::colP(b), qm0 + soff(st), t > 0);      // dK += dS^T Q
        tc::mma_commit(BAR(C::QD_EMPTY + st));
        if (t + 2 < n) ok = sp(t + 2);
    }
    tc::mma_commit(BAR(C::ACC_FULL));
    tc::mma_commit(BAR(C::DONE));
    wait(C::DONE, 0);
}

template <int HD>
__device__ void kv_softmax(const BwdTcParams &p, const KvWork &w, uint32_t bar0, uint32_t tmem, const float *vec) {
    using C = KvCfg<HD>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = warp >> 2;
    const uint32_t row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    const uint32_t j = w.k0 + row;
    const bool row_ok = j < p.Lr;
    const uint32_t kpos = pos32(p.split, w.s, min(j, p.Lr - 1), p.c, p.rd);
    uint32_t sa = 0, se = p.L;  // the key's sample (packed sequences)
    if (p.cu) sample_bounds(p.cu, p.nseq, kpos, p.L, sa, se);
    const float sl2 = p.scale_log2;
    const uint32_t n = kv_count_tiles(p, w);
    QIter it;
    qiter_init(p, w, it);
    uint32_t r_cur = 0xffffffffu, i0 = 0, i1 = 0;
    bool ok = true;
    for (uint32_t t = 0; t < n && !it.done; ++t) {
        const uint32_t st = t % C::kStages, b = t & 1u;
        if (it.r != r_cur) {
            // the query rows of rank r that see this key: [i0, i1)
            r_cur = it.r;
            i0 = before32(p.split, p.causal ? kpos : sa, r_cur, p.c, p.rd);
            i1 = before32(p.split, se, r_cur, p.c, p.rd);
        }
        ok = tc::mbar_wait(BAR(C::SP_FULL + b), (t >> 1) & 1u, p.status, USP_ERR_TIMEOUT, kWaitNs) &&
             tc::mbar_wait(BAR(C::QD_FULL + st), (t / C::kStages) & 1u, p.status, USP_ERR_TIMEOUT, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t tS = tmem + lane_off + C::colS(b) + 32u * half;
        const uint32_t tP = tmem + lane_off + C::colP(b) + 32u * half;
        uint32_t sv[32], dpv[32];
        tc::tmem_ld32(tS, sv);
        tc::tmem_ld32(tP, dpv);
        float l2[32], dd[32];
        const float4 *l4 = reinterpret_cast<const float4 *>(vec + st * kT + 32 * half);
        const float4 *d4 = reinterpret_cast<const float4 *>(vec + C::kStages * kT + st * kT + 32 * half);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 a = l4[q], d = d4[q];
            l2[4 * q] = a.x; l2[4 * q + 1] = a.y; l2[4 * q + 2] = a.z; l2[4 * q + 3] = a.w;
            dd[4 * q] = d.x; dd[4 * q + 1] = d.y; dd[4 * q + 2] = d.z; dd[4 * q + 3] = d.w;
        }
        // query row it.n * 64 + 32 half + e sees key j iff it lies in [i0, i1)
        const int c0 = (int)(it.n * kT) + 32 * half;
        const int lo = (int)i0 - c0;
        const int hi = row_ok ? (int)i1 - c0 : 0;
        tc::tmem_ld_wait();
        uint32_t pk[16], dk[16];
        p_ds_half(sv, dpv, l2, dd, sl2, lo, hi, pk, dk);
        tc::tmem_st16(tS, pk);
        tc::tmem_st16(tP, dk);
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(BAR(C::P_FULL + b));
        qiter_advance(p, w, it);
    }
    if (!ok) return;
    // epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (times the softmax scale)
    __nv_bfloat16 *dst = (half == 0 ? p.g1 : p.g0) + ((size_t)w.kv_row0 + j) * HD;
    if (n == 0) {
        if (row_ok)
            for (int oc = 0; oc < HD / 32; ++oc) store_zero32(dst + oc * 32);
        return;
    }
    ok = tc::mbar_wait(BAR(C::ACC_FULL), 0, p.status, USP_ERR_TIMEOUT, kWaitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return;
    tc::fence_after_sync();
    const uint32_t tA = tmem + lane_off + (half == 0 ? 0u : (uint32_t)HD);
    const float mul = half == 0 ? 1.f : p.scale;
#pragma unroll 1
    for (int oc = 0; oc < HD / 32; ++oc) {
        uint32_t o[32];
        tc::tmem_ld32(tA + oc * 32, o);
        tc::tmem_ld_wait();
        if (row_ok) store_row32(dst + oc * 32, o, mul);
    }
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkv_kernel(const __grid_constant__ BwdTcParams p) {
    using C = KvCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    const uint32_t bar0 = sbase + C::kBar;
    float *vec = reinterpret_cast<float *>(smem + C::kVec);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kTmemSlot);
    volatile uint32_t *skip_flag = tmem_slot + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        *skip_flag = (*reinterpret_cast<volatile int *>(p.status) != 0) ? 1u : 0u;
        tc::mbar_init(bar0 + 8u * C::KV_FULL, 1);
        for (int s = 0; s < C::kStages; ++s) {
            tc::mbar_init(bar0 + 8u * (C::QD_FULL + s), 32);
            tc::mbar_init(bar0 + 8u * (C::QD_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(bar0 + 8u * (C::SP_FULL + b), 1);
            tc::mbar_init(bar0 + 8u * (C::P_FULL + b), 8);
        }
        tc::mbar_init(bar0 + 8u * C::ACC_FULL, 1);
        tc::mbar_init(bar0 + 8u * C::DONE, 1);
        tc::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tc::prefetch_tmap(&p.t_big0);
        tc::prefetch_tmap(&p.t_big1);
        tc::prefetch_tmap(&p.t_small0);
        tc::prefetch_tmap(&p.t_small1);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *skip_flag != 0;
    const KvWork w = kv_decode(p);
    if (!skip) {
        if (warp == kProducerWarp) {
            kv_producer<HD>(p, w, sbase, bar0, vec);
        } else if (warp == kMmaWarp) {
            if (lane == 0) kv_mma<HD>(p, w, sbase, bar0, tmem);
            __syncwarp();
        } else if (warp < 8) {
            kv_softmax<HD>(p, w, bar0, tmem, vec);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ================================================================================================
// dq kernel
// ================================================================================================
// The dq kernel streams 128-key tiles (N = 128 products run at the full rate, N = 64 ones do not).
constexpr int kKT = 128;

template <int HD> struct QCfg : Lay<HD> {
    using Y = Lay<HD>;
    static constexpr int kKS = HD == 128 ? 3 : 4;           // K stages: K(t) for S(t) and dQ(t), K(t+2) for S(t+2)
    static constexpr int kVS = HD == 128 ? 2 : 3;           // V stages: V(t+1) for dP(t+1)
    static constexpr int kQ = 0;
    static constexpr int kDo = Y::kBigTile;
    static constexpr int kK = 2 * Y::kBigTile;              // K stage s at kK + s * kBigTile
    static constexpr int kV = kK + kKS * Y::kBigTile;       // V stage s at kV + s * kBigTile
    static constexpr int kBar = kV + kVS * Y::kBigTile;
    static constexpr int QO_FULL = 0;
    static constexpr int K_FULL = 1;                         // [kKS]
    static constexpr int K_EMPTY = K_FULL + kKS;             // [kKS]
    static constexpr int V_FULL = K_EMPTY + kKS;             // [kVS]
    static constexpr int V_EMPTY = V_FULL + kVS;             // [kVS]
    static constexpr int S_FULL = V_EMPTY + kVS;             // [2]: S_b complete
    static constexpr int DP_FULL = S_FULL + 2;               // dP complete
    static constexpr int DP_FREE = DP_FULL + 1;              // dP loaded by the softmax (8 warps)
    static constexpr int DS_FULL = DP_FREE + 1;              // [2]: dS written over S_b (8 warps)
    static constexpr int ACC_FULL = DS_FULL + 2;
    static constexpr int DONE = ACC_FULL + 1;
    static constexpr int kNumBars = DONE + 1;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kSmemBytes = kTmemSlot + 16 + 1024;
    // TMEM: dQ [0, hd), S_0 [hd, hd + 128), S_1 [hd + 128, hd + 256), dP [hd + 256, hd + 384)
    __device__ static constexpr uint32_t colS(int b) { return (uint32_t)HD + 128u * (uint32_t)b; }
    __device__ static constexpr uint32_t colP() { return (uint32_t)HD + 256u; }
};
static_assert(QCfg<128>::kSmemBytes <= 232448, "dq kernel shared memory");

// register split of the dq kernel (setmaxnreg): a softmax thread holds 64 S and 64 dP values
constexpr int kQSoftmaxRegs = 208, kQControlRegs = 88;
static_assert(2 * kQSoftmaxRegs + kQControlRegs == 504, "the launch's 168 registers per thread");

struct QWork {
    uint32_t r, u, h, b, kh, q0;
    uint32_t q_row0;  // row of local query 0 of (r, u, h, b) in q / dout / dq / lse / delta
    uint32_t qpos_min, qpos_max;
    uint32_t sa_first, se_last;  // sample start of the first row, sample end of the last (packed)
};

__device__ __forceinline__ QWork q_decode(const BwdTcParams &p) {
    QWork w;
    const uint32_t inner = p.ud * p.Hl * p.bs;
    const uint32_t outer = blockIdx.x / inner;
    uint32_t in = blockIdx.x % inner;
    w.h = in % p.Hl;
    in /= p.Hl;
    w.b = in % p.bs;
    w.u = in / p.bs;
    if (p.lpt) {
        // zigzag, heaviest first: global 128-row blocks from the end of the sequence
        const uint32_t per_chunk = p.c / 128;
        const uint32_t gp = 2 * p.rd * per_chunk - 1 - outer;
        const uint32_t a = gp / per_chunk, off = (gp % per_chunk) * 128;
        w.r = a < p.rd ? a : 2 * p.rd - 1 - a;
        w.q0 = (a < p.rd ? 0 : p.c) + off;
    } else if (p.split == USP_SPLIT_BASIC) {
        const uint32_t gp = p.rd * p.ntiles - 1 - outer;
        w.r = gp / p.ntiles;
        w.q0 = (gp % p.ntiles) * 128;
    } else {
        w.r = outer % p.rd;
        w.q0 = (p.ntiles - 1 - outer / p.rd) * 128;
    }
    w.kh = w.h / p.G;
    w.q_row0 = (((w.r * p.ud + w.u) * p.Hl + w.h) * p.bs + w.b) * p.Lr;
    w.qpos_min = pos32(p.split, w.r, w.q0, p.c, p.rd);
    w.qpos_max = pos32(p.split, w.r, min(w.q0 + 127, p.Lr - 1), p.c, p.rd);
    w.sa_first = 0;
    w.se_last = p.L;
    if (p.cu) {
        uint32_t a, e;
        sample_bounds(p.cu, p.nseq, w.qpos_min, p.L, w.sa_first, e);
        sample_bounds(p.cu, p.nseq, w.qpos_max, p.L, a, w.se_last);
    }
    return w;
}

// KV tiles of 128 keys over the ring steps (Fig. 1 order), over the rows of rank s that some query
// of the tile sees: from the first row's sample start to the last row's visible limit
struct KIter {
    uint32_t t, s, kt, nkt;
    bool done;
};

__device__ __forceinline__ void q_key_range(const BwdTcParams &p, const QWork &w, uint32_t s, uint32_t &kt0,
                                            uint32_t &kt1) {
    const uint32_t lo = before32(p.split, w.sa_first, s, p.c, p.rd);
    const uint32_t hi = p.causal ? vis32(p.split, w.qpos_max, s, p.c, p.rd) : before32(p.split, w.se_last, s, p.c, p.rd);
    kt0 = lo / kKT;
    kt1 = hi > lo ? (hi + kKT - 1) / kKT : kt0;
}

__device__ __forceinline__ void kiter_step(const BwdTcParams &p, const QWork &w, KIter &it) {
    it.s = (w.r + p.rd - it.t) % p.rd;
    q_key_range(p, w, it.s, it.kt, it.nkt);
}

__device__ __forceinline__ void kiter_init(const BwdTcParams &p, const QWork &w, KIter &it) {
    it.t = 0;
    it.done = false;
    kiter_step(p, w, it);
    while (it.kt >= it.nkt) {
        if (++it.t >= p.rd) {
            it.done = true;
            return;
        }
        kiter_step(p, w, it);
    }
}

__device__ __forceinline__ void kiter_advance(const BwdTcParams &p, const QWork &w, KIter &it) {
    if (++it.kt < it.nkt) return;
    do {
        if (++it.t >= p.rd) {
            it.done = true;
            return;
        }
        kiter_step(p, w, it);
    } while (it.kt >= it.nkt);
}

__device__ __forceinline__ uint32_t q_count_tiles(const BwdTcParams &p, const QWork &w) {
    uint32_t n = 0;
    for (uint32_t t = 0; t < p.rd; ++t) {
        uint32_t kt0, kt1;
        q_key_range(p, w, (w.r + p.rd - t) % p.rd, kt0, kt1);
        n += kt1 - kt0;
    }
    return n;
}

// Q and dout once; then per KV tile K into a K stage and V into a V stage, each waiting only for its
// own stage to be released (K after dQ(t), V after dP(t))
template <int HD>
__device__ void q_producer(const BwdTcParams &p, const QWork &w, uint32_t sbase, uint32_t bar0) {
    using C = QCfg<HD>;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    auto wait = [&](int bar, uint32_t parity) {
        return tc::mbar_wait(BAR(bar), parity, p.status, USP_ERR_TIMEOUT, kWaitNs);
    };
    tc::mbar_arrive_expect_tx(BAR(C::QO_FULL), 2 * C::kBigTile);
    for (int bx = 0; bx < C::kBoxes; ++bx) {
        tc::tma_load_2d(sbase + C::kQ + bx * C::kBigBox, &p.t_big0, bx * 64, (int32_t)(w.q_row0 + w.q0),
                        BAR(C::QO_FULL));
        tc::tma_load_2d(sbase + C::kDo + bx * C::kBigBox, &p.t_big1, bx * 64, (int32_t)(w.q_row0 + w.q0),
                        BAR(C::QO_FULL));
    }
    KIter it;
    kiter_init(p, w, it);
    uint32_t t = 0, kf = 0, vf = 0;
    bool ok = true;
    while (!it.done) {
        const uint32_t kv_row = (((it.s * p.ud + w.u) * p.Hkl + w.kh) * p.bs + w.b) * p.Lr + it.kt * kKT;
        const uint32_t ks = t % C::kKS, vs = t % C::kVS;
        if (!(ok = wait(C::K_EMPTY + ks, ((t / C::kKS) & 1u) ^ 1u))) break;
        tc::mbar_arrive_expect_tx(BAR(C::K_FULL + ks), C::kBigTile);
        for (int bx = 0; bx < C::kBoxes; ++bx)
            tc::tma_load_2d(sbase + C::kK + ks * C::kBigTile + bx * C::kBigBox, &p.t_small0, bx * 64, (int32_t)kv_row,
                            BAR(C::K_FULL + ks));
        ++kf;
        if (!(ok = wait(C::V_EMPTY + vs, ((t / C::kVS) & 1u) ^ 1u))) break;
        tc::mbar_arrive_expect_tx(BAR(C::V_FULL + vs), C::kBigTile);
        for (int bx = 0; bx < C::kBoxes; ++bx)
            tc::tma_load_2d(sbase + C::kV + vs * C::kBigTile + bx * C::kBigBox, &p.t_small1, bx * 64, (int32_t)kv_row,
                            BAR(C::V_FULL + vs));
        ++vf;
        ++t;
        kiter_advance(p, w, it);
    }
    if (!ok) {
        // drain the copies this thread issued before the CTA exits
        wait(C::QO_FULL, 0);
        for (uint32_t f = kf > C::kKS ? kf - C::kKS : 0; f < kf; ++f) wait(C::K_FULL + f % C::kKS, (f / C::kKS) & 1u);
        for (uint32_t f = vf > C::kVS ? vf - C::kVS : 0; f < vf; ++f) wait(C::V_FULL + f % C::kVS, (f / C::kVS) & 1u);
    }
}

// S_b(t) = Q K(t)^T into one of two S buffers, dP(t) = dout V(t)^T into the one dP buffer as soon
// as the softmax has loaded dP(t-1), dQ += dS(t) K(t) (A = dS, written as bf16 over S_b) once the
// softmax has written it, then S(t+2) over the same S buffer (issued after dQ(t), so it cannot
// overwrite dS(t) before dQ(t) has read it).
template <int HD>
__device__ void q_mma(const BwdTcParams &p, const QWork &w, uint32_t sbase, uint32_t bar0, uint32_t tmem) {
    using C = QCfg<HD>;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    auto wait = [&](int bar, uint32_t parity) {
        return tc::mbar_wait(BAR(bar), parity, p.status, USP_ERR_TIMEOUT, kWaitNs);
    };
    const uint32_t n = q_count_tiles(p, w);
    const uint64_t qdesc = tc::sw128_desc(sbase + C::kQ, 16, 1024);
    const uint64_t odesc = tc::sw128_desc(sbase + C::kDo, 16, 1024);
    const uint64_t kdesc = tc::sw128_desc(sbase + C::kK, 16, 1024);              // K-major view of K
    const uint64_t kmdesc = tc::sw128_desc(sbase + C::kK, C::kBigBox, 1024);     // MN-major view of K
    const uint64_t vdesc = tc::sw128_desc(sbase + C::kV, 16, 1024);
    constexpr uint32_t idS = tc::idesc_bf16_f32(128, kKT, 0, 0);
    constexpr uint32_t idQ = tc::idesc_bf16_f32(128, HD, 0, 1);
    auto toff = [](uint32_t st) { return (uint64_t)((st * C::kBigTile) >> 4); };
    auto kofs = [](int kk) { return (uint64_t)(((kk / 4) * C::kBigBox + (kk % 4) * 32) >> 4); };
    auto issue_s = [&](uint32_t t) {
        const uint32_t ks = t % C::kKS;
        if (!wait(C::K_FULL + ks, (t / C::kKS) & 1u)) return false;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
            tc::mma_ss(tmem + C::colS(t & 1u), qdesc + kofs(kk), kdesc + toff(ks) + kofs(kk), idS, kk > 0 ? 1u : 0u);
        tc::mma_commit(BAR(C::S_FULL + (t & 1u)));
        return true;
    };
    auto issue_dp = [&](uint32_t t) {
        const uint32_t vs = t % C::kVS;
        if (!wait(C::V_FULL + vs, (t / C::kVS) & 1u)) return false;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
            tc::mma_ss(tmem + C::colP(), odesc + kofs(kk), vdesc + toff(vs) + kofs(kk), idS, kk > 0 ? 1u : 0u);
        tc::mma_commit(BAR(C::DP_FULL));
        tc::mma_commit(BAR(C::V_EMPTY + vs));
        return true;
    };
    bool ok = wait(C::QO_FULL, 0);
    if (ok && n > 0) ok = issue_s(0) && issue_dp(0);
    if (ok && n > 1) ok = issue_s(1);
    for (uint32_t t = 0; ok && t < n; ++t) {
        const uint32_t b = t & 1u, ks = t % C::kKS;
        // the softmax of tile t has loaded dP(t): compute dP(t+1) while it works
        if (t + 1 < n) {
            if (!(ok = wait(C::DP_FREE, t & 1u))) break;
            tc::fence_after_sync();
            if (!(ok = issue_dp(t + 1))) break;
        }
        if (!(ok = wait(C::DS_FULL + b, (t >> 1) & 1u))) break;
        tc::fence_after_sync();
        // dQ += dS(t) K(t): k-step kk reads keys [16 kk, 16 kk + 16), packed by the softmax at TMEM
        // column 64 (kk / 4) + 8 (kk % 4) of S_b; K viewed MN-major (N = hd), 16 keys = 2048 bytes
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk)
            tc::mma_ts(tmem, tmem + C::colS(b) + 64u * (kk / 4) + 8u * (kk % 4),
                       kmdesc + toff(ks) + (uint64_t)((kk * 2048) >> 4), idQ, (t > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(BAR(C::K_EMPTY + ks));
        if (t + 2 < n) ok = issue_s(t + 2);
    }
    tc::mma_commit(BAR(C::ACC_FULL));
    tc::mma_commit(BAR(C::DONE));
    wait(C::DONE, 0);
}

// two warpgroups, each owning keys [64 h, 64 h + 64) of every 128-key tile and one thread per query
// row: load S and dP, release dP, compute dS = P (dP - D) with P = exp2(S scale log2e - lse log2e)
// (0 outside the row's visible key range), write dS as bf16 over its own half of S
template <int HD>
__device__ void q_softmax(const BwdTcParams &p, const QWork &w, uint32_t bar0, uint32_t tmem) {
    using C = QCfg<HD>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = warp >> 2;
    const uint32_t row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    const uint32_t i = w.q0 + row;
    const bool row_ok = i < p.Lr;
    const uint32_t qpos = pos32(p.split, w.r, min(i, p.Lr - 1), p.c, p.rd);
    uint32_t sa = 0, se = p.L;  // the row's sample (packed sequences)
    if (p.cu) sample_bounds(p.cu, p.nseq, qpos, p.L, sa, se);
    const float lse2 = row_ok ? p.lse[w.q_row0 + i] * kLog2e : 0.f;
    const float di = row_ok ? p.delta[w.q_row0 + i] : 0.f;
    float l2[32], dd[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        l2[e] = lse2;
        dd[e] = di;
    }
    const float sl2 = p.scale_log2;
    const uint32_t n = q_count_tiles(p, w);
    KIter it;
    kiter_init(p, w, it);
    uint32_t s_cur = 0xffffffffu, nvis = 0, klo = 0;
    bool ok = true;
    for (uint32_t t = 0; t < n && !it.done; ++t) {
        const uint32_t b = t & 1u;
        if (it.s != s_cur) {
            // the rows of rank s this query sees: [klo, nvis)
            s_cur = it.s;
            nvis = p.causal ? vis32(p.split, qpos, s_cur, p.c, p.rd) : before32(p.split, se, s_cur, p.c, p.rd);
            klo = before32(p.split, sa, s_cur, p.c, p.rd);
        }
        ok = tc::mbar_wait(BAR(C::S_FULL + b), (t >> 1) & 1u, p.status, USP_ERR_TIMEOUT, kWaitNs) &&
             tc::mbar_wait(BAR(C::DP_FULL), t & 1u, p.status, USP_ERR_TIMEOUT, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t tS = tmem + lane_off + C::colS(b) + 64u * half;
        const uint32_t tP = tmem + lane_off + C::colP() + 64u * half;
        uint32_t sv[2][32], dpv[2][32];
        tc::tmem_ld32(tS, sv[0]);
        tc::tmem_ld32(tS + 32, sv[1]);
        tc::tmem_ld32(tP, dpv[0]);
        tc::tmem_ld32(tP + 32, dpv[1]);
        tc::tmem_ld_wait();
        // dP is in registers: the next dP may be computed into the buffer
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(BAR(C::DP_FREE));
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            // key it.kt * 128 + 64 half + 32 c + e is visible iff it lies in the row's range [klo, nvis)
            const int c0 = (int)(it.kt * kKT) + 64 * half + 32 * c;
            const int lo = (int)klo - c0;
            const int hi = row_ok ? (int)nvis - c0 : 0;
            uint32_t pk[16], dk[16];
            p_ds_half(sv[c], dpv[c], l2, dd, sl2, lo, hi, pk, dk);
            tc::tmem_st16(tS + 16 * c, dk);
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(BAR(C::DS_FULL + b));
        kiter_advance(p, w, it);
    }
    if (!ok) return;
    // epilogue: warpgroup 0 writes dq columns [0, hd/2), warpgroup 1 [hd/2, hd), times the scale
    __nv_bfloat16 *dst = p.g0 + ((size_t)w.q_row0 + i) * HD;
    if (n == 0) {
        if (row_ok)
            for (int oc = half * HD / 64; oc < (half + 1) * HD / 64; ++oc) store_zero32(dst + oc * 32);
        return;
    }
    ok = tc::mbar_wait(BAR(C::ACC_FULL), 0, p.status, USP_ERR_TIMEOUT, kWaitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return;
    tc::fence_after_sync();
#pragma unroll 1
    for (int oc = half * HD / 64; oc < (half + 1) * HD / 64; ++oc) {
        uint32_t o[32];
        tc::tmem_ld32(tmem + lane_off + oc * 32, o);
        tc::tmem_ld_wait();
        if (row_ok) store_row32(dst + oc * 32, o, p.scale);
    }
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdTcParams p) {
    using C = QCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    const uint32_t bar0 = sbase + C::kBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kTmemSlot);
    volatile uint32_t *skip_flag = tmem_slot + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        *skip_flag = (*reinterpret_cast<volatile int *>(p.status) != 0) ? 1u : 0u;
        tc::mbar_init(bar0 + 8u * C::QO_FULL, 1);
        for (int s = 0; s < C::kKS; ++s) {
            tc::mbar_init(bar0 + 8u * (C::K_FULL + s), 1);
            tc::mbar_init(bar0 + 8u * (C::K_EMPTY + s), 1);
        }
        for (int s = 0; s < C::kVS; ++s) {
            tc::mbar_init(bar0 + 8u * (C::V_FULL + s), 1);
            tc::mbar_init(bar0 + 8u * (C::V_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(bar0 + 8u * (C::S_FULL + b), 1);
            tc::mbar_init(bar0 + 8u * (C::DS_FULL + b), 8);
        }
        tc::mbar_init(bar0 + 8u * C::DP_FULL, 1);
        tc::mbar_init(bar0 + 8u * C::DP_FREE, 8);
        tc::mbar_init(bar0 + 8u * C::ACC_FULL, 1);
        tc::mbar_init(bar0 + 8u * C::DONE, 1);
        tc::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tc::prefetch_tmap(&p.t_big0);
        tc::prefetch_tmap(&p.t_big1);
        tc::prefetch_tmap(&p.t_small0);
        tc::prefetch_tmap(&p.t_small1);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *skip_flag != 0;
    const QWork w = q_decode(p);
    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kQControlRegs));
        if (!skip) {
            if (warp == kProducerWarp && lane == 0) q_producer<HD>(p, w, sbase, bar0);
            else if (warp == kMmaWarp && lane == 0) q_mma<HD>(p, w, sbase, bar0, tmem);
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kQSoftmaxRegs));
        if (!skip) q_softmax<HD>(p, w, bar0, tmem);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------------
template <typename Kern>
int prepare(Kern kern, int smem, bool &done) {
    if (done) return USP_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return USP_ERR_CUDA;
    done = true;
    return USP_OK;
}

template <int HD>
int launch_typed(BwdTcParams &kv, BwdTcParams &q, uint32_t grid_kv, uint32_t grid_q, cudaStream_t s) {
    static bool set_kv[64] = {}, set_q[64] = {};
    static std::mutex set_mu;  // host threads may make their first launch at the same time
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return USP_ERR_CUDA;
    std::unique_lock<std::mutex> lk(set_mu);
    int rc = prepare(attn_bwd_dkv_kernel<HD>, KvCfg<HD>::kSmemBytes, set_kv[dev]);
    if (rc) return rc;
    if (!set_q[dev]) {
        // setmaxnreg.inc can only be granted from registers the launch holds: refuse a build whose
        // register count would make the split wait
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, attn_bwd_dq_kernel<HD>) != cudaSuccess) return USP_ERR_CUDA;
        if ((long)fa.numRegs * kThreads < 2L * 128 * kQSoftmaxRegs + 128L * kQControlRegs) return USP_ERR_UNSUPPORTED;
    }
    if ((rc = prepare(attn_bwd_dq_kernel<HD>, QCfg<HD>::kSmemBytes, set_q[dev]))) return rc;
    lk.unlock();
    attn_bwd_dkv_kernel<HD><<<grid_kv, kThreads, KvCfg<HD>::kSmemBytes, s>>>(kv);
    attn_bwd_dq_kernel<HD><<<grid_q, kThreads, QCfg<HD>::kSmemBytes, s>>>(q);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace

int launch_attn_bwd_tc(const BwdArgs &a, cudaStream_t s) {
    const AttnArgs &f = a.f;
    const DeviceInfo *di = device_info();
    if (!di) return USP_ERR_CUDA;
    BwdTcParams base{};
    base.lse = f.lse;
    base.delta = a.delta;
    base.status = di->status;
    base.bs = (uint32_t)f.bs;
    base.rd = (uint32_t)f.rd;
    base.ud = (uint32_t)f.ud;
    base.Lr = (uint32_t)(f.L / f.rd);
    base.c = (uint32_t)(f.L / (2 * f.rd));
    base.Hl = (uint32_t)(f.hq / f.ud);
    base.Hkl = (uint32_t)heads_per_rank(f.hkv, f.ud);
    base.G = (uint32_t)(f.hq / f.hkv);
    base.ntiles = (base.Lr + 127) / 128;
    base.causal = f.causal;
    base.split = f.split;
    base.lpt = (f.split == USP_SPLIT_ZIGZAG && base.c % 128 == 0) ? 1 : 0;
    base.scale = f.scale;
    base.scale_log2 = f.scale * kLog2e;
    base.cu = f.cu;
    base.nseq = (uint32_t)f.nseq;
    base.L = (uint32_t)f.L;
    const uint64_t q_rows = (uint64_t)f.hq * f.bs * f.L;
    const uint64_t kv_rows = (uint64_t)base.Hkl * f.ud * f.bs * f.L;
    BwdTcParams kv = base, q = base;
    if (!make_tmap(&kv.t_big0, f.k, kv_rows, f.hd, 128) || !make_tmap(&kv.t_big1, f.v, kv_rows, f.hd, 128) ||
        !make_tmap(&kv.t_small0, f.q, q_rows, f.hd, kT) || !make_tmap(&kv.t_small1, a.dout, q_rows, f.hd, kT) ||
        !make_tmap(&q.t_big0, f.q, q_rows, f.hd, 128) || !make_tmap(&q.t_big1, a.dout, q_rows, f.hd, 128) ||
        !make_tmap(&q.t_small0, f.k, kv_rows, f.hd, kKT) || !make_tmap(&q.t_small1, f.v, kv_rows, f.hd, kKT))
        return USP_ERR_CUDA;
    kv.g0 = static_cast<__nv_bfloat16 *>(a.dk);
    kv.g1 = static_cast<__nv_bfloat16 *>(a.dv);
    q.g0 = static_cast<__nv_bfloat16 *>(a.dq);
    const uint64_t grid_kv = (uint64_t)base.rd * base.ntiles * base.ud * base.Hkl * base.bs;
    const uint64_t grid_q = (uint64_t)base.rd * base.ntiles * base.ud * base.Hl * base.bs;
    if (grid_kv == 0 || grid_q == 0) return USP_OK;
    if (grid_kv >= (1ull << 31) || grid_q >= (1ull << 31)) return USP_ERR_UNSUPPORTED;
    return f.hd == 128 ? launch_typed<128>(kv, q, (uint32_t)grid_kv, (uint32_t)grid_q, s)
                       : launch_typed<64>(kv, q, (uint32_t)grid_kv, (uint32_t)grid_q, s);
}

}  // namespace usp
