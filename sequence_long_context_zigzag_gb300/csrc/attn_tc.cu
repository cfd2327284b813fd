// attn_tc.cu -- bf16 LoadBalance-RingAttention forward on the 5th-generation tensor cores (sm_103a).
//
// What it computes (USP review, Algorithm 1 step 4; Context-Parallel page, section 先弄清楚 and
// Fig. 1): for every virtual ring rank r, Ulysses rank u, local query head h and batch b, the rows of
// rank r's zigzag-local sequence attend to the KV blocks of ring ranks (r - t) mod rd for
// t = 0 .. rd-1 in that order, under the causal mask on global positions; the per-block partials are
// folded by the log-sum-exp merge. Here the merge is the online-softmax rescale inside one pass, so
// no partial ever leaves the chip (the fused-merge epilogue). USP_MODE_STEP / USP_MODE_ACCUM run a
// single ring step and write its partial, or merge it into (out, lse) in the epilogue.
//
// Kernel design. A unit of work is 256 query rows = two 128-row Q tiles of one (r, u, h, b). The
// kernel is persistent: one CTA per SM (or on fewer SMs, when a caller keeps some free for another
// stream's kernels) walks a static list of units, and its roles run through the
// units without a CTA-wide barrier, so one unit's epilogue overlaps the next unit's Q / K loads and
// first S products. Units are numbered by cost, heaviest first, or in super-groups of heads whose
// directions alternate (see decode_work), and round k of gridDim.x units goes to the CTAs in order for
// even k and in reverse for odd k, which balances rounds whose costs fall or rise steadily.
//   warp 8      TMA producer: Q0, Q1 once per unit (after both issuers' last S product of the previous
//               unit has completed); K and V tiles (128 keys x hd) through a ring of stages that runs on
//               across units.
//   warps 9, 10 MMA issuers, one thread per Q tile i: S_i = Q_i K^T and O_i += P_i V on tcgen05
//               (kind::f16, bf16 in, fp32 accumulators in tensor memory), issue order PV_i(j),
//               S_i(j+1), so the tensor core works on one tile while the other tile's softmax runs.
//   warps 0-3   softmax of Q tile 0, warps 4-7 softmax of Q tile 1: one thread per query row reads
//               its S row from TMEM, masks partial tiles, updates the running max with a lazy
//               rescale (O and l are rescaled only when the max grows by more than 2^8), writes
//               P = 2^(S*scale*log2e - m) as bf16 back into TMEM (the A operand of the PV MMA), and
//               at the end of each unit normalises O and writes out (bf16) and lse (fp32), then hands
//               O's columns back to the issuer for the next unit.
//   warp 11     holds no role; with warps 8-10 it forms the control warpgroup that hands registers
//               to the softmax warpgroups (setmaxnreg).
//   TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+hd) O1 [256+hd, 256+2hd); P_i aliases S_i.
// The causal structure is exploited per (Q tile, KV tile) pair from global positions: tiles wholly
// after the queries are skipped (never loaded), tiles wholly before are unmasked, the rest are
// masked per element with a per-row key limit (the zigzag map is increasing inside a rank, so the
// keys a row sees in a rank's block are a prefix of it).
// Every wait is bounded (2 s): on expiry the kernel records USP_ERR_TIMEOUT in the device status
// word, drains what it has in flight and returns.
#include <cuda.h>

#include <algorithm>

#include "tc_common.cuh"
#include "tc_ptx.cuh"
#include "usp_device.cuh"
#include "usp_internal.cuh"

namespace usp {
namespace {

constexpr int kM = 128;  // query rows per tile
constexpr int kN = 128;  // keys per tile
// one softmax warpgroup per Q tile (two per tile, 640 threads with a shared-memory max exchange per
// KV tile, measured 6% slower on GB300)
constexpr int kSoftmaxWarps = 8;               // 2 Q tiles x 4 warps
constexpr int kWarps = kSoftmaxWarps + 4;      // plus the control warpgroup
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;    // issues Q tile 0's MMAs; allocates and frees tensor memory
constexpr int kMmaWarp1 = kSoftmaxWarps + 2;   // issues Q tile 1's MMAs
// Register split per warpgroup (setmaxnreg). The launch grants kThreads x kLaunchRegs registers; the
// softmax warpgroups take 2 x 128 x kSoftmaxRegs and the control warpgroup keeps
// 128 x kControlRegs, together exactly the launch's registers, so the increase can always be granted.
constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8;
constexpr int kSoftmaxRegs = 208;
constexpr int kControlRegs = kLaunchRegs * kWarps / 4 - 2 * kSoftmaxRegs;
static_assert(kSoftmaxRegs % 8 == 0 && kControlRegs % 8 == 0 && kControlRegs >= 24 && kControlRegs <= 256 &&
                  2 * kSoftmaxRegs + kControlRegs == kLaunchRegs * kWarps / 4,
              "register split must use exactly the launch's registers");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// packed samples: cu_seqlens entries kept in shared memory (every role decodes every unit, with four
// binary searches, and every softmax thread searches its row's sample); longer arrays are read from
// global memory
constexpr int kCuCache = 4096;
constexpr uint64_t kSuperGroupKV = 64ull << 20;  // K/V bytes per super-group of units (launch_attn_tc)
constexpr uint64_t kSingleGroupKV = 128ull << 20;  // largest group K/V numbered as its own super-group
constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

template <int HD> struct Cfg {
    static constexpr int kBoxes = HD / 64;            // 64-column (128-byte) TMA boxes per row
    static constexpr int kBoxBytes = kM * 128;         // 128 rows x 128 bytes
    static constexpr int kTileBytes = kM * HD * 2;     // 128 rows x hd bf16
    static constexpr int kStages = (HD == 128) ? 2 : 4;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + 2 * kTileBytes;
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kBar = kV + kStages * kTileBytes;
    // barrier indices (K and V stages have their own barriers: K(j+1) is needed one softmax earlier
    // than V(j+1), and K's stage frees earlier, so split barriers give the copies more lead time)
    static constexpr int Q_FULL = 0;
    static constexpr int K_FULL = 1;
    static constexpr int K_EMPTY = K_FULL + kStages;
    static constexpr int V_FULL = K_EMPTY + kStages;
    static constexpr int V_EMPTY = V_FULL + kStages;
    static constexpr int S_FULL = V_EMPTY + kStages;  // [2]
    static constexpr int P_FULL = S_FULL + 2;         // [2]
    static constexpr int O_FULL = P_FULL + 2;         // [2]
    static constexpr int DONE = O_FULL + 2;           // [2]
    static constexpr int TURN = DONE + 2;             // [2]: issuer i may issue its next burst
    static constexpr int Q_EMPTY = TURN + 2;          // both issuers' S products of a unit are done
    static constexpr int O_EMPTY = Q_EMPTY + 1;       // [2]: the softmax has read O_i of a unit
    static constexpr int kNumBars = O_EMPTY + 2;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    // at kTmemSlot: tensor memory address, skip flag; then (packed samples only) a copy of cu_seqlens
    static constexpr int kCu = kTmemSlot + 16;
    // epilogue staging of the packed-sample kernel, after the cu_seqlens copy: one slot per softmax
    // warp (32 rows x 64 bytes)
    static constexpr int kStgSlot = 32 * 64;
    static constexpr int kStgBytes = kSoftmaxWarps * kStgSlot;
    __host__ __device__ static constexpr int stg_offset(bool pk) {
        return (kCu + (pk ? kCuCache * 4 : 0) + 127) / 128 * 128;
    }
    __device__ static constexpr uint32_t colS(int i) { return 128u * (uint32_t)i; }
    __device__ static constexpr uint32_t colO(int i) { return 256u + (uint32_t)(HD * i); }
};

struct TcParams {
    CUtensorMap tq, tk, tv;
    __nv_bfloat16 *out;
    float *lse;
    int *status;
    uint32_t bs, Lr, c, rd, ud, Hl, Hkl, npairs, units;
    uint32_t Gl, ngroups, nouter, sg, sg_flip;  // unit numbering: see decode_work
    int causal, mode, step, lpt, split, ring_rank_only;
    float scale_log2;
    const int32_t *cu;  // packed samples' cumulative lengths, or nullptr
    uint32_t nseq, L;
};

// The work of one unit and the walk over its KV tiles (identical in every role). Positions and row
// indices fit in 31 bits (the entry point rejects larger tensors), so 32-bit arithmetic is used.
struct Work {
    uint32_t r, u, hl, b, kh;
    uint32_t q_row_base;  // row of local row 0 of (r, u, hl, b) in q / out / lse
    uint32_t q0[2];       // first local row of each Q tile
    bool valid[2];
    uint32_t qpos_min[2], qpos_max[2];
    uint32_t sa_first[2], sa_last[2];  // sample start of the tile's first / last row (0 unless packed)
    uint32_t se_first[2], se_last[2];  // sample end (one past) of the first / last row (L unless packed)
    int t_begin, t_end;
};

struct Tile {
    uint32_t s, kt;
    uint32_t kv_row;  // first row of the tile in k / v
    bool act[2];      // the Q tile needs this KV tile
    bool full[2];     // every key of the tile is visible to every row of the Q tile
    bool first;       // first tile of its unit (set by cursor_next only)
};

// Per ring step, the keys of rank s's block visible to a row form a range of its rows [lo, hi)
// (every split's position map increases with the row; packed samples cut the range at the row's
// sample start). Over the rows of a Q tile both ends are non-decreasing, so the tile's first and last
// rows bound them: lomin / lomax are the first / last row's lo, nlo / nhi their hi.
struct TileIter {
    int t;
    uint32_t kt, nkt, s;
    uint32_t nhi[2], nlo[2];
    uint32_t lomin[2], lomax[2];
};

// The k-th unit of this CTA: round k covers units [k G, (k + 1) G) of the numbering (decode_work), in
// CTA order for even k and in reverse order for odd k. False when the CTA has no k-th unit.
__device__ __forceinline__ bool unit_index(const TcParams &p, uint32_t k, uint32_t &x) {
    const uint32_t G = gridDim.x, b = blockIdx.x;
    x = k * G + ((k & 1u) ? G - 1 - b : b);
    return x < p.units;
}

// sample_bounds on the shared-memory copy of cu_seqlens (at shared address cu_s)
__device__ __forceinline__ void sample_bounds_smem(uint32_t cu_s, uint32_t nseq, uint32_t g, uint32_t L, uint32_t &a,
                                                   uint32_t &e) {
    auto ld = [](uint32_t addr) {
        int32_t v;
        asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr));
        return v;
    };
    uint32_t lo = 0, hi = nseq;
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (ld(cu_s + 4u * mid) <= (int32_t)g) lo = mid;
        else hi = mid;
    }
    const int32_t a0 = ld(cu_s + 4u * lo), e0 = ld(cu_s + 4u * lo + 4u);
    a = (a0 < 0 || (uint32_t)a0 > g) ? (a0 < 0 ? 0u : g) : (uint32_t)a0;
    e = (e0 <= (int32_t)g) ? g + 1 : ((uint32_t)e0 > L ? L : (uint32_t)e0);
}

// the sample [a, e) of global position g: from the shared-memory copy when cu_seqlens fits there
// (cu_s != 0), else from global memory
__device__ __forceinline__ void sample_of(const TcParams &p, uint32_t cu_s, uint32_t g, uint32_t &a, uint32_t &e) {
    if (cu_s) sample_bounds_smem(cu_s, p.nseq, g, p.L, a, e);
    else sample_bounds(p.cu, p.nseq, g, p.L, a, e);
}

// cu_s: shared address of the cu_seqlens copy, or 0 (packed samples only)
template <bool PK>
__device__ __forceinline__ Work decode_work(const TcParams &p, uint32_t cu_s, uint32_t x) {
    Work w;
    // Units that read the same K/V (one local KV head of one Ulysses rank and batch element: a
    // group of Gl query heads x nouter 256-row blocks) are numbered in super-groups of sg groups.
    // Inside a super-group the blocks go by cost (outer), each block across the super-group's heads.
    // sg is all groups unless a smaller super-group saves DRAM traffic (launch_attn_tc): then
    // the SMs work on one or two heads at a time and read their K/V from L2 after the first touch,
    // even though the static schedule lets units that share K/V drift apart in time.
    const uint32_t per_group = p.nouter * p.Gl;
    const uint32_t sgi = x / (p.sg * per_group);  // super-group
    const uint32_t g0 = sgi * p.sg;
    const uint32_t n = min(p.sg, p.ngroups - g0);
    const uint32_t xl = x - g0 * per_group;
    uint32_t outer = xl / (n * p.Gl);
    const uint32_t rem = xl % (n * p.Gl);
    // super-groups alternate in direction, the last one heaviest first (sg_flip = parity of the
    // super-group count minus one): where one super-group ends and the next begins, the costs meet
    // at the same level (both light or both heavy), which keeps the snake's pairs of rounds balanced
    // across the boundary; a heavy-to-light order throughout put two of the heaviest units on the
    // CTAs at the end of the boundary's round
    if ((sgi ^ p.sg_flip) & 1u) outer = p.nouter - 1 - outer;
    const uint32_t grp = g0 + rem / p.Gl;
    w.b = grp % p.bs;
    const uint32_t uk = grp / p.bs;  // u Hkl + kh
    w.kh = uk % p.Hkl;
    w.u = uk / p.Hkl;
    w.hl = w.kh * p.Gl + rem % p.Gl;
    uint32_t qp;
    if (p.ring_rank_only > 0) {
        // one ring rank's share only, its later rows (more keys) first
        w.r = (uint32_t)(p.ring_rank_only - 1);
        qp = p.npairs - 1 - outer;
    } else if (p.lpt) {
        // zigzag, heaviest first: global 256-row blocks from the end of the sequence to its start
        const uint32_t per_chunk = p.c / 256;
        const uint32_t gp = 2 * p.rd * per_chunk - 1 - outer;
        const uint32_t a = gp / per_chunk;
        const uint32_t off = (gp % per_chunk) * 256;
        w.r = a < p.rd ? a : 2 * p.rd - 1 - a;
        qp = ((a < p.rd) ? off : p.c + off) / 256;
    } else if (p.split == USP_SPLIT_BASIC) {
        // contiguous blocks: the last rank's last rows are the heaviest
        const uint32_t gp = p.rd * p.npairs - 1 - outer;
        w.r = gp / p.npairs;
        qp = gp % p.npairs;
    } else {
        // stripe (and zigzag with chunks that are not whole 256-row blocks): later rows first
        w.r = outer % p.rd;
        qp = p.npairs - 1 - outer / p.rd;
    }
    w.q_row_base = (((w.r * p.ud + w.u) * p.Hl + w.hl) * p.bs + w.b) * p.Lr;
    for (int i = 0; i < 2; ++i) {
        w.q0[i] = qp * 256 + i * 128;
        w.valid[i] = w.q0[i] < p.Lr;
        const uint32_t last = min(w.q0[i] + 127, p.Lr - 1);
        w.qpos_min[i] = pos32(p.split, w.r, min(w.q0[i], p.Lr - 1), p.c, p.rd);
        w.qpos_max[i] = pos32(p.split, w.r, last, p.c, p.rd);
        w.sa_first[i] = w.sa_last[i] = 0;
        w.se_first[i] = w.se_last[i] = p.L;
        if constexpr (PK) {
            sample_of(p, cu_s, w.qpos_min[i], w.sa_first[i], w.se_first[i]);
            sample_of(p, cu_s, w.qpos_max[i], w.sa_last[i], w.se_last[i]);
        }
    }
    w.t_begin = p.mode == USP_MODE_FUSED ? 0 : p.step;
    w.t_end = p.mode == USP_MODE_FUSED ? (int)p.rd : p.step + 1;
    return w;
}

template <bool PK>
__device__ __forceinline__ void iter_setup(const TcParams &p, const Work &w, TileIter &it) {
    it.s = (w.r + p.rd - (uint32_t)it.t) % p.rd;
    uint32_t mx = 0, mn = 0xffffffffu;
    for (int i = 0; i < 2; ++i) {
        if (!w.valid[i]) {
            it.nhi[i] = 0;
            it.nlo[i] = 0;
            it.lomin[i] = 0;
            it.lomax[i] = 0;
            continue;
        }
        if (p.causal) {
            it.nhi[i] = vis32(p.split, w.qpos_max[i], it.s, p.c, p.rd);
            it.nlo[i] = vis32(p.split, w.qpos_min[i], it.s, p.c, p.rd);
        } else {
            it.nhi[i] = PK ? before32(p.split, w.se_last[i], it.s, p.c, p.rd) : p.Lr;
            it.nlo[i] = PK ? before32(p.split, w.se_first[i], it.s, p.c, p.rd) : p.Lr;
        }
        it.lomin[i] = PK ? before32(p.split, w.sa_first[i], it.s, p.c, p.rd) : 0u;
        it.lomax[i] = PK ? before32(p.split, w.sa_last[i], it.s, p.c, p.rd) : 0u;
        if (it.nhi[i] > it.lomin[i]) {
            mx = max(mx, it.nhi[i]);
            mn = min(mn, it.lomin[i]);
        }
    }
    it.nkt = (uint32_t)((mx + kN - 1) / kN);
    it.kt = mn == 0xffffffffu ? it.nkt : mn / kN;
}

template <bool PK>
__device__ __forceinline__ void iter_init(const TcParams &p, const Work &w, TileIter &it) {
    if constexpr (PK) {
        // the first iter_next call sets up ring step t_begin: one inlined copy of iter_setup, which
        // pays for packed samples (units of a few tiles) and not for long units
        it.t = w.t_begin - 1;
        it.kt = 0;
        it.nkt = 0;
    } else {
        it.t = w.t_begin;
        iter_setup<PK>(p, w, it);
    }
}

// the next KV tile that at least one Q tile of the unit needs (packed samples can leave gaps between
// the two Q tiles' key ranges; every role skips the same tiles)
template <bool PK>
__device__ __forceinline__ bool iter_next(const TcParams &p, const Work &w, TileIter &it, Tile &tl) {
    for (;;) {
        while (it.kt >= it.nkt) {
            if (++it.t >= w.t_end) return false;
            iter_setup<PK>(p, w, it);
        }
        if constexpr (PK) {
            for (int i = 0; i < 2; ++i) {
                tl.act[i] = it.kt * kN < it.nhi[i] && (it.kt + 1) * kN > it.lomin[i];
                tl.full[i] = (it.kt + 1) * kN <= it.nlo[i] && it.kt * kN >= it.lomax[i];
            }
            if (tl.act[0] || tl.act[1]) break;
            ++it.kt;
        } else {
            // one sample: the key ranges start at row 0 and the Q tile with the larger range is active
            for (int i = 0; i < 2; ++i) {
                tl.act[i] = it.kt * kN < it.nhi[i];
                tl.full[i] = (it.kt + 1) * kN <= it.nlo[i];
            }
            break;
        }
    }
    tl.s = it.s;
    tl.kt = it.kt;
    tl.kv_row = (((it.s * p.ud + w.u) * p.Hkl + w.kh) * p.bs + w.b) * p.Lr + it.kt * kN;
    ++it.kt;
    return true;
}

// The CTA's tiles as one stream across its units (units without a tile are passed over), for the
// MMA issuers, whose bursts run from one unit into the next.
struct Cursor {
    uint32_t k;  // sequence number of the next unit to open
    bool live;   // w / it hold an open unit
    Work w;
    TileIter it;
};

template <bool PK>
__device__ __forceinline__ bool cursor_next(const TcParams &p, uint32_t cu_s, Cursor &c, Tile &tl) {
    bool first = false;
    while (!(c.live && iter_next<PK>(p, c.w, c.it, tl))) {
        uint32_t x;
        if (!unit_index(p, c.k, x)) {
            c.live = false;
            return false;
        }
        ++c.k;
        c.w = decode_work<PK>(p, cu_s, x);
        iter_init<PK>(p, c.w, c.it);
        c.live = true;
        first = true;
    }
    tl.first = first;
    return true;
}

// ------------------------------------------------------------------------------------------------
// roles
// ------------------------------------------------------------------------------------------------
// One thread issues every copy: per unit Q0 and Q1 (once both issuers have finished the previous
// unit's S products, which read Q), then for each KV tile K into a K stage and V into a V stage, each
// waiting only for its own stage to be released. Stage fills are counted across units.
template <int HD, bool PK>
__device__ void producer_role(const TcParams &p, uint32_t cu_s, uint32_t sbase, uint32_t bar0) {
    using C = Cfg<HD>;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    auto wait = [&](int bar, uint32_t parity) {
        return tc::mbar_wait(BAR(bar), parity, p.status, USP_ERR_TIMEOUT, kWaitLimitNs);
    };
    const uint32_t sQ = sbase + C::kQ, sK = sbase + C::kK, sV = sbase + C::kV;
    uint32_t kfills = 0, vfills = 0, nq = 0;  // stage fills and Q loads issued
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
        uint32_t x;
        if (!unit_index(p, k, x)) break;
        const Work w = decode_work<PK>(p, cu_s, x);
        TileIter it;
        iter_init<PK>(p, w, it);
        Tile tl;
        bool first = true;  // a unit without a tile loads nothing
        while (ok && iter_next<PK>(p, w, it, tl)) {
            if (first) {
                first = false;
                if (nq > 0 && !(ok = wait(C::Q_EMPTY, (nq - 1) & 1u))) break;
                tc::mbar_arrive_expect_tx(BAR(C::Q_FULL), 2 * C::kTileBytes);
                for (int i = 0; i < 2; ++i)
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        tc::tma_load_2d(sQ + i * C::kTileBytes + bx * C::kBoxBytes, &p.tq, bx * 64,
                                        (int32_t)(w.q_row_base + w.q0[i]), BAR(C::Q_FULL));
                ++nq;
            }
            const uint32_t st = kfills % C::kStages;
            const uint32_t ph = ((kfills / C::kStages) & 1u) ^ 1u;
            if (!(ok = wait(C::K_EMPTY + st, ph))) break;
            tc::mbar_arrive_expect_tx(BAR(C::K_FULL + st), C::kTileBytes);
            for (int bx = 0; bx < C::kBoxes; ++bx)
                tc::tma_load_2d(sK + st * C::kTileBytes + bx * C::kBoxBytes, &p.tk, bx * 64, (int32_t)tl.kv_row,
                                BAR(C::K_FULL + st));
            ++kfills;
            if (!(ok = wait(C::V_EMPTY + st, ph))) break;
            tc::mbar_arrive_expect_tx(BAR(C::V_FULL + st), C::kTileBytes);
            for (int bx = 0; bx < C::kBoxes; ++bx)
                tc::tma_load_2d(sV + st * C::kTileBytes + bx * C::kBoxBytes, &p.tv, bx * 64, (int32_t)tl.kv_row,
                                BAR(C::V_FULL + st));
            ++vfills;
        }
    }
    if (!ok) {
        // drain: wait (bounded) for the copies this thread issued, so none lands after the CTA exits
        // (Q loads are issued one at a time, each after the previous one was consumed)
        if (nq > 0) wait(C::Q_FULL, (nq - 1) & 1u);
        for (uint32_t f = kfills > C::kStages ? kfills - C::kStages : 0; f < kfills; ++f)
            wait(C::K_FULL + f % C::kStages, (f / C::kStages) & 1u);
        for (uint32_t f = vfills > C::kStages ? vfills - C::kStages : 0; f < vfills; ++f)
            wait(C::V_FULL + f % C::kStages, (f / C::kStages) & 1u);
    }
}

// The descriptors' start-address field holds (shared address >> 4) in its low 14 bits; shared
// memory is below 256 KB, so adding (byte offset >> 4) to a base descriptor moves its start address.
template <int HD>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc) {
    using C = Cfg<HD>;
    constexpr uint32_t idS = tc::idesc_bf16_f32(kM, kN, 0, 0);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint64_t koff = (uint64_t)(((kk / 4) * C::kBoxBytes + (kk % 4) * 32) >> 4);
        tc::mma_ss(d_tmem, qdesc + koff, kdesc + koff, idS, kk > 0 ? 1u : 0u);
    }
}

template <int HD>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc, uint32_t accumulate) {
    // B = V viewed as (N = hd) x (K = keys), MN-major: 64-column blocks C::kBoxBytes apart (LBO),
    // 8-key groups 1024 bytes apart (SBO); 16 keys per MMA = 2048 bytes.
    constexpr uint32_t idO = tc::idesc_bf16_f32(kM, HD, 0, 1);
#pragma unroll
    for (int kk = 0; kk < kN / 16; ++kk)
        tc::mma_ts(d_tmem, p_tmem + kk * 8, vdesc + (uint64_t)((kk * 2048) >> 4), idO,
                   (accumulate || kk > 0) ? 1u : 0u);
}

// One thread per Q tile issues that tile's MMAs and commits, and the two take turns: S_0(0) | S_1(0) |
// PV_0(0) S_0(1) | PV_1(0) S_1(1) | PV_0(1) S_0(2) | ... Each burst waits for its operands (V, P, K)
// first and for its turn last, so it issues the moment the other burst has been queued: the tensor
// core always has one issuer's burst running while the other issuer waits, and the two Q tiles stay
// half a period apart (one tile's softmax runs while the other tile's MMAs run).
// Per burst j of issuer i, in order: PV_i(j) [commit: V stage of tile j released by this issuer],
// S_i(j+1) [commits: S_i ready, K stage of tile j+1 released by this issuer]. Stage barriers count one
// release from each issuer. PV_i(j) and S_i(j+1) come from the same thread, so the tensor core runs
// them in that order: S_i(j+1) overwrites the columns where P_i(j) lives only after PV_i(j) has read
// them, and when the softmax sees S_i(j+1) complete, PV_i(j) is complete too (which makes its
// in-place rescale of O_i safe). The tcgen05 fence follows only the wait on the softmax threads' P
// (TMA completion is ordered by the mbarrier).
// The bursts run on from one unit into the next. At the start of the burst of a unit's last tile each
// issuer commits to Q_EMPTY (its S products of the unit were all issued in earlier bursts; once both
// issuers' commits arrive, the producer loads the next unit's Q), and after the last PV it commits
// O_FULL_i.
// When tile j+1 opens a new unit, S_i(j+1) leaves the turn order: issuer i releases its turn after
// PV_i(j), waits for the new Q and K(j+1) and issues S_i(j+1) at once, without waiting for the other
// issuer's last PV (which waits for the other softmax's last tile), so the unit's first S products
// run while the softmaxes finish the old unit; both issuers skip the turn there, so their turn
// counts stay equal. The first PV of a unit waits for O_EMPTY_i, the softmax's read-out of the
// previous unit's O_i. A Q tile without a visible key in a unit takes no O_FULL / O_EMPTY round (the
// softmax skips it too).
template <int HD, bool PK>
__device__ void mma_role(const TcParams &p, uint32_t cu_s, uint32_t sbase, uint32_t bar0, uint32_t tmem, int i) {
    using C = Cfg<HD>;
    auto BAR = [&](int k) { return bar0 + 8u * k; };
    auto wait = [&](int bar, uint32_t parity) {
        return tc::mbar_wait(BAR(bar), parity, p.status, USP_ERR_TIMEOUT, kWaitLimitNs);
    };
    const uint32_t sQ = sbase + C::kQ, sK = sbase + C::kK, sV = sbase + C::kV;
    // base descriptors: this Q tile and stage 0 of K / V (K-major: LBO unused, SBO = 8 rows x 128 B;
    // V as MN-major: LBO = next 64-column block, SBO = next 8-key group)
    const uint64_t qdesc = tc::sw128_desc(sQ + (uint32_t)i * C::kTileBytes, 16, 1024);
    const uint64_t kdesc0 = tc::sw128_desc(sK, 16, 1024);
    const uint64_t vdesc0 = tc::sw128_desc(sV, C::kBoxBytes, 1024);
    auto stage_off = [](uint32_t st) { return (uint64_t)((st * C::kTileBytes) >> 4); };
    const uint32_t tS = tmem + C::colS(i), tO = tmem + C::colO(i);
    const int barS = C::S_FULL + i, barP = C::P_FULL + i;
    const int my_turn = C::TURN + i, other_turn = C::TURN + (1 - i);
    // turn phases: issuer 0's burst j (j >= 0) waits for issuer 1's burst j-1; issuer 1's burst j
    // (j >= -1) waits for issuer 0's burst j
    uint32_t turns = 0;
    auto take_turn = [&]() { return wait(my_turn, (turns++) & 1u); };
    // S_i of tile t from K stage st, and this issuer's release of the stage
    auto s_burst = [&](const Tile &t, uint32_t st) {
        if (i ? t.act[1] : t.act[0]) {
            issue_s<HD>(tS, qdesc, kdesc0 + stage_off(st));
            tc::mma_commit(BAR(barS));
        }
        tc::mma_commit(BAR(C::K_EMPTY + st));
    };
    Cursor cs;
    cs.k = 0;
    cs.live = false;
    Tile cur, nxt;
    bool have = cursor_next<PK>(p, cu_s, cs, cur);
    bool ok = true;
    uint32_t pc = 0, started = 0;  // P waits; a PV of the current unit has been issued
    uint32_t nq = 0, no = 0;       // Q loads consumed; O_i read-outs handed to the softmax
    uint32_t j = 0;                // tiles of the stream (stage ring position)
    if (have) {
        ok = wait(C::Q_FULL, 0) && wait(C::K_FULL + 0, 0);
        nq = 1;
        if (ok && i == 1) ok = take_turn();
        if (ok) {
            s_burst(cur, 0);
            tc::mbar_arrive(BAR(other_turn));
        }
    }
    while (ok && have) {
        const bool have_n = cursor_next<PK>(p, cu_s, cs, nxt);
        const bool last = !have_n || nxt.first;      // tile j is the last of its unit
        const bool boundary = have_n && nxt.first;  // tile j+1 opens a new unit
        const uint32_t st = j % C::kStages, ph = (j / C::kStages) & 1u;
        const uint32_t stn = (j + 1) % C::kStages, phn = ((j + 1) / C::kStages) & 1u;
        const bool act = i ? cur.act[1] : cur.act[0];
        if (last) tc::mma_commit(BAR(C::Q_EMPTY));  // this issuer's S products of the unit are issued
        // operands first: every issuer waits for a stage's fill before releasing it, even when its Q
        // tile skips the tile, so neither issuer can release fill f + kStages before the producer has
        // refilled the stage (which needs both releases of fill f): the shared release barrier never
        // runs ahead
        if (!(ok = wait(C::V_FULL + st, ph))) break;
        if (act && !(ok = wait(barP, pc & 1u))) break;
        if (act && !started && no > 0 && !(ok = wait(C::O_EMPTY + i, (no - 1) & 1u))) break;
        if (have_n && !boundary && !(ok = wait(C::K_FULL + stn, phn))) break;
        if (!(ok = take_turn())) break;
        if (act) {
            ++pc;
            tc::fence_after_sync();
            issue_pv<HD>(tO, tS, vdesc0 + stage_off(st), started);
            started = 1;
        }
        tc::mma_commit(BAR(C::V_EMPTY + st));  // this issuer no longer reads V(j)
        if (last) {
            if (started) {
                tc::mma_commit(BAR(C::O_FULL + i));
                ++no;
            }
            started = 0;
        }
        if (have_n && !boundary) s_burst(nxt, stn);
        tc::mbar_arrive(BAR(other_turn));
        if (boundary) {
            if (!(ok = wait(C::Q_FULL, nq & 1u))) break;
            ++nq;
            if (!(ok = wait(C::K_FULL + stn, phn))) break;
            s_burst(nxt, stn);
        }
        cur = nxt;
        have = have_n;
        ++j;
    }
    if (!ok) tc::mbar_arrive(BAR(other_turn));  // let the other issuer reach its own bounded exit
    // every MMA of this issuer has finished before tensor memory is released
    tc::mma_commit(BAR(C::DONE + i));
    wait(C::DONE + i, 0);
}

// The issuer of the packed-sample kernel: the same products, commits and turn order as mma_role,
// written so that the unit decode (cursor_next) and the S burst are each inlined once, and with the
// stream's first S products outside the turn order like every later unit's. Packed samples cross a
// unit boundary every few tiles, so the boundary code runs often and its size and latency count:
// measured on GB300 this version is 9-12% faster for packed samples of 1024 to 4096 tokens, while
// for long units (one sample) it is 1.5-2% slower than mma_role, which stays there.
template <int HD, bool PK>
__device__ void mma_role_pk(const TcParams &p, uint32_t cu_s, uint32_t sbase, uint32_t bar0, uint32_t tmem, int i) {
    using C = Cfg<HD>;
    auto BAR = [&](int k) { return bar0 + 8u * k; };
    auto wait = [&](int bar, uint32_t parity) {
        return tc::mbar_wait(BAR(bar), parity, p.status, USP_ERR_TIMEOUT, kWaitLimitNs);
    };
    const uint32_t sQ = sbase + C::kQ, sK = sbase + C::kK, sV = sbase + C::kV;
    // base descriptors: this Q tile and stage 0 of K / V (K-major: LBO unused, SBO = 8 rows x 128 B;
    // V as MN-major: LBO = next 64-column block, SBO = next 8-key group)
    const uint64_t qdesc = tc::sw128_desc(sQ + (uint32_t)i * C::kTileBytes, 16, 1024);
    const uint64_t kdesc0 = tc::sw128_desc(sK, 16, 1024);
    const uint64_t vdesc0 = tc::sw128_desc(sV, C::kBoxBytes, 1024);
    auto stage_off = [](uint32_t st) { return (uint64_t)((st * C::kTileBytes) >> 4); };
    const uint32_t tS = tmem + C::colS(i), tO = tmem + C::colO(i);
    const int barS = C::S_FULL + i, barP = C::P_FULL + i;
    const int my_turn = C::TURN + i, other_turn = C::TURN + (1 - i);
    // turn phases: issuer 0's burst j (j >= 0) waits for issuer 1's burst j-1; issuer 1's burst j
    // (j >= -1) waits for issuer 0's burst j
    uint32_t turns = 0;
    auto take_turn = [&]() { return wait(my_turn, (turns++) & 1u); };
    // S_i of tile t from K stage st, and this issuer's release of the stage
    auto s_burst = [&](const Tile &t, uint32_t st) {
        if (i ? t.act[1] : t.act[0]) {
            issue_s<HD>(tS, qdesc, kdesc0 + stage_off(st));
            tc::mma_commit(BAR(barS));
        }
        tc::mma_commit(BAR(C::K_EMPTY + st));
    };
    Cursor cs;
    cs.k = 0;
    cs.live = false;
    Tile cur, nxt;
    bool have = false;             // cur holds tile j of the stream
    bool ok = true;
    uint32_t pc = 0, started = 0;  // P waits; a PV of the current unit has been issued
    uint32_t nq = 0, no = 0;       // Q loads consumed; O_i read-outs handed to the softmax
    uint32_t j = 0;                // tiles of the stream (stage ring position)
    // The stream's first S products are outside the turn order like every unit's first ones; issuer
    // 1's empty "burst -1" lets issuer 0's burst 0 go first.
    if (i == 1) tc::mbar_arrive(BAR(other_turn));
    // One loop pass per tile j: PV_i(j) in the turn order, then S_i(j+1); cursor_next and the S
    // burst are inlined once each.
    while (ok) {
        const bool have_n = cursor_next<PK>(p, cu_s, cs, nxt);
        const bool boundary = have_n && nxt.first;  // tile j+1 opens a unit (the stream's first tile too)
        const uint32_t jn = have ? j + 1 : 0;       // stream index of nxt
        const uint32_t stn = jn % C::kStages, phn = (jn / C::kStages) & 1u;
        bool turn_after_s = false;                   // S_i(j+1) is part of this burst
        if (have) {
            const bool last = !have_n || nxt.first;  // tile j is the last of its unit
            const uint32_t st = j % C::kStages, ph = (j / C::kStages) & 1u;
            const bool act = i ? cur.act[1] : cur.act[0];
            if (last) tc::mma_commit(BAR(C::Q_EMPTY));  // this issuer's S products of the unit are issued
            // operands first: every issuer waits for a stage's fill before releasing it, even when its
            // Q tile skips the tile, so neither issuer can release fill f + kStages before the producer
            // has refilled the stage (which needs both releases of fill f): the shared release barrier
            // never runs ahead
            if (!(ok = wait(C::V_FULL + st, ph))) break;
            if (act && !(ok = wait(barP, pc & 1u))) break;
            if (act && !started && no > 0 && !(ok = wait(C::O_EMPTY + i, (no - 1) & 1u))) break;
            if (have_n && !boundary && !(ok = wait(C::K_FULL + stn, phn))) break;
            if (!(ok = take_turn())) break;
            if (act) {
                ++pc;
                tc::fence_after_sync();
                issue_pv<HD>(tO, tS, vdesc0 + stage_off(st), started);
                started = 1;
            }
            tc::mma_commit(BAR(C::V_EMPTY + st));  // this issuer no longer reads V(j)
            if (last) {
                if (started) {
                    tc::mma_commit(BAR(C::O_FULL + i));
                    ++no;
                }
                started = 0;
            }
            turn_after_s = have_n && !boundary;
            if (!turn_after_s) tc::mbar_arrive(BAR(other_turn));
        }
        if (!have_n) break;
        if (boundary) {
            if (!(ok = wait(C::Q_FULL, nq & 1u))) break;
            ++nq;
            if (!(ok = wait(C::K_FULL + stn, phn))) break;
        }
        s_burst(nxt, stn);
        if (turn_after_s) tc::mbar_arrive(BAR(other_turn));
        cur = nxt;
        have = true;
        j = jn;
    }
    if (!ok) tc::mbar_arrive(BAR(other_turn));  // let the other issuer reach its own bounded exit
    // every MMA of this issuer has finished before tensor memory is released
    tc::mma_commit(BAR(C::DONE + i));
    wait(C::DONE + i, 0);
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// columns at or beyond the row's key limit (relative to the tile) get score -inf
__device__ __forceinline__ void mask_chunk(uint32_t (&r)[32], int col0, int lim_local) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
        if (col0 + e >= lim_local) r[e] = __float_as_uint(-INFINITY);
}

// packed samples: columns outside the row's visible range [lo_local, lim_local) get score -inf
__device__ __forceinline__ void mask_chunk2(uint32_t (&r)[32], int col0, int lo_local, int lim_local) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
        if (col0 + e >= lim_local || col0 + e < lo_local) r[e] = __float_as_uint(-INFINITY);
}

__device__ __forceinline__ float chunk_max(const uint32_t (&r)[32]) {
    float a = u2f(r[0]), b = u2f(r[1]);
#pragma unroll
    for (int e = 2; e < 30; e += 4) {
        a = tc::max3(a, u2f(r[e]), u2f(r[e + 1]));
        b = tc::max3(b, u2f(r[e + 2]), u2f(r[e + 3]));
    }
    a = tc::max3(a, u2f(r[30]), u2f(r[31]));
    return fmaxf(a, b);
}

// P = 2^(s * scale*log2e - mb) for one 32-column chunk: accumulate the row sum, pack to bf16 pairs
__device__ __forceinline__ void chunk_exp(const uint32_t (&r)[32], uint64_t sl22, uint64_t nmb2, uint64_t &sacc,
                                          uint32_t (&pk)[16]) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const uint64_t y = tc::fma2(tc::pack2(u2f(r[2 * e]), u2f(r[2 * e + 1])), sl22, nmb2);
        float y0, y1;
        tc::unpack2(y, y0, y1);
        const float p0 = tc::ex2(y0), p1 = tc::ex2(y1);
        sacc = tc::add2(sacc, tc::pack2(p0, p1));
        pk[e] = float2_to_bf16x2(p0, p1);
    }
}

// The softmax of Q tile i: one thread per query row (TMEM lane = row). Per KV tile each thread reads
// its S row from TMEM in one round trip, and O and l are rescaled only when the running max grows by
// more than 2^8 (lazy rescale: exact, because the final normalisation uses the same stale max).
// P = 2^(s*scale*log2e - m) is packed to bf16 and written over the start of S, where the PV MMA
// reads it as its A operand. A failed (timed-out) wait in any lane makes the whole warp leave (the
// warps of the tile then fail their own next waits, which the recorded status ends quickly).
// One call handles one unit; ns (S tiles consumed) and no (O read-outs) run on across units, as the
// barrier phases do. Returns false after a failed wait.
template <int HD, bool PK>
__device__ __forceinline__ bool softmax_unit(const TcParams &p, uint32_t cu_s, const Work &w, uint32_t bar0,
                                             uint32_t tmem, uint32_t stg, int i, uint32_t &ns, uint32_t &no) {
    using C = Cfg<HD>;
    constexpr int kCh = 4;  // 32-column chunks of an S row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wq = warp & 3;
    const uint32_t row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + 128u * (uint32_t)i;
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(HD * i);
    const uint32_t barS = bar0 + 8u * (C::S_FULL + i);
    const uint32_t barP = bar0 + 8u * (C::P_FULL + i);
    const uint32_t barO = bar0 + 8u * (C::O_FULL + i);
    const uint32_t barOE = bar0 + 8u * (C::O_EMPTY + i);
    const uint32_t q0 = i ? w.q0[1] : w.q0[0];
    const bool valid = i ? w.valid[1] : w.valid[0];
    const uint32_t row_local = q0 + row;
    const bool row_ok = valid && row_local < p.Lr;
    const uint32_t qpos_row = pos32(p.split, w.r, min(row_local, p.Lr - 1), p.c, p.rd);
    uint32_t sa_row = 0, se_row = p.L;  // the row's sample (packed sequences)
    if constexpr (PK) sample_of(p, cu_s, qpos_row, sa_row, se_row);
    const float sl2 = p.scale_log2;
    const uint64_t sl22 = tc::pack2(sl2, sl2);

    float m_used = -INFINITY, l = 0.f;
    uint32_t n_act = 0;
    bool ok = true;
    TileIter it;
    iter_init<PK>(p, w, it);
    Tile tl;
    uint32_t s_cur = 0xffffffffu;
    uint32_t lim = 0, lim_lo = 0;
    while (iter_next<PK>(p, w, it, tl)) {
        const bool act = i ? tl.act[1] : tl.act[0];
        if (!act) continue;
        const bool full = i ? tl.full[1] : tl.full[0];
        if (tl.s != s_cur) {
            s_cur = tl.s;
            lim = p.causal ? vis32(p.split, qpos_row, s_cur, p.c, p.rd)
                           : (PK ? before32(p.split, se_row, s_cur, p.c, p.rd) : p.Lr);
            if constexpr (PK) lim_lo = before32(p.split, sa_row, s_cur, p.c, p.rd);
        }
        ok = tc::mbar_wait(barS, ns & 1u, p.status, USP_ERR_TIMEOUT, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        uint32_t sr[kCh][32];
        float mx = -INFINITY;
        if (ok) {
            tc::fence_after_sync();
#pragma unroll
            for (int cc = 0; cc < kCh; ++cc) tc::tmem_ld32(tS + cc * 32, sr[cc]);
            tc::tmem_ld_wait();
            if (!full) {
                const int ll = (int)lim - (int)(tl.kt * kN);
                const int lim_local = ll < 0 ? 0 : (ll > kN ? kN : ll);
                if constexpr (PK) {
                    const int lo_local = (int)lim_lo - (int)(tl.kt * kN);
#pragma unroll
                    for (int cc = 0; cc < kCh; ++cc) mask_chunk2(sr[cc], cc * 32, lo_local, lim_local);
                } else {
#pragma unroll
                    for (int cc = 0; cc < kCh; ++cc) mask_chunk(sr[cc], cc * 32, lim_local);
                }
            }
#pragma unroll
            for (int cc = 0; cc < kCh; ++cc) mx = fmaxf(mx, chunk_max(sr[cc]));
            mx *= sl2;
        }
        if (!ok) break;
        const bool need = mx > m_used + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
            const float m_new = fmaxf(m_used, mx);
            const float alpha = need ? tc::ex2(m_used - m_new) : 1.f;  // 0 on the first visible tile
            if (need) m_used = m_new;
            if (n_act > 0) {
                // O, 32 columns at a time (the S row is still live in registers)
#pragma unroll 1
                for (int oc = 0; oc < HD / 32; ++oc) {
                    uint32_t o[32];
                    tc::tmem_ld32(tO + oc * 32, o);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(u2f(o[e]) * alpha);
                    tc::tmem_st32(tO + oc * 32, o);
                }
            }
            l *= alpha;
        }
        const float mb = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t nmb2 = tc::pack2(-mb, -mb);
        uint64_t sacc = tc::pack2(0.f, 0.f);
#pragma unroll
        for (int cc = 0; cc < kCh; ++cc) {
            uint32_t pk[16];
            chunk_exp(sr[cc], sl22, nmb2, sacc, pk);
            tc::tmem_st16(tS + cc * 16, pk);
        }
        float s0, s1;
        tc::unpack2(sacc, s0, s1);
        l += s0 + s1;
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(barP);
        ++n_act;
        ++ns;
    }
    if (!ok) return false;
    // ---- epilogue: normalise, merge (ACCUM), store ------------------
    const size_t grow = (size_t)w.q_row_base + row_local;
    const float lse_cur = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
    float w_old = 0.f, w_new = 1.f, lse_out = lse_cur;
    if (p.mode == USP_MODE_ACCUM && row_ok) merge_weights(p.lse[grow], lse_cur, w_old, w_new, lse_out);
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16 *orow = p.out + grow * HD;
    constexpr int kOc = HD / 32;  // 32-column chunks of O
    if (n_act > 0) {
        ok = tc::mbar_wait(barO, no & 1u, p.status, USP_ERR_TIMEOUT, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        ++no;
        tc::fence_after_sync();
        // all of O's columns in one round trip, then O_i goes back to the issuer
        uint32_t o[kOc][32];
#pragma unroll
        for (int oc = 0; oc < kOc; ++oc) tc::tmem_ld32(tO + oc * 32, o[oc]);
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(barOE);
        if (PK && p.mode != USP_MODE_ACCUM) {
            // Packed samples (short units, where the epilogue recurs every few tiles): each lane packs
            // its row's 32-column chunk (64 bytes) into the warp's staging slot, 16-byte
            // pieces swizzled by (row / 2) mod 4 so that neither the row-wise writes nor the
            // column-wise reads conflict on banks; then every store instruction of the warp writes 8
            // whole 64-byte row segments (4 lanes per row), 8 lines instead of one per lane. Measured
            // on GB300: packed samples of 1024 tokens 15% faster; one long sample 1.5% slower (there
            // the epilogue is a few per cent of the time and the kernel's code layout moves), so the
            // one-sample kernel keeps the per-row stores below.
            const uint32_t wrow0 = q0 + (uint32_t)wq * 32u;  // local row of the warp's first row
            const size_t gbase = (size_t)w.q_row_base + wrow0;
            const uint32_t rd_r = (uint32_t)lane >> 2, rd_c = (uint32_t)lane & 3u;
#pragma unroll
            for (int oc = 0; oc < kOc; ++oc) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = float2_to_bf16x2(u2f(o[oc][2 * e]) * inv_l, u2f(o[oc][2 * e + 1]) * inv_l);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    st_shared_v4(stg + (uint32_t)lane * 64u + (((uint32_t)c4 ^ (((uint32_t)lane >> 1) & 3u)) << 4),
                                 pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
                __syncwarp();
#pragma unroll
                for (int it8 = 0; it8 < 4; ++it8) {
                    const uint32_t r = (uint32_t)it8 * 8u + rd_r;
                    const uint4 x = ld_shared_v4(stg + r * 64u + ((rd_c ^ ((r >> 1) & 3u)) << 4));
                    if (valid && wrow0 + r < p.Lr)
                        *reinterpret_cast<uint4 *>(p.out + (gbase + r) * HD + oc * 32 + rd_c * 8) = x;
                }
                __syncwarp();
            }
        } else if (row_ok) {
#pragma unroll
            for (int oc = 0; oc < kOc; ++oc) {
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = u2f(o[oc][e]) * inv_l;
                uint4 *dst = reinterpret_cast<uint4 *>(orow + oc * 32);
                if (p.mode == USP_MODE_ACCUM) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 old = dst[q];
                        const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const float2 f = bf16x2_to_float2(ow[h]);
                            v[q * 8 + 2 * h] = w_old * f.x + w_new * v[q * 8 + 2 * h];
                            v[q * 8 + 2 * h + 1] = w_old * f.y + w_new * v[q * 8 + 2 * h + 1];
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 pkd;
                    pkd.x = float2_to_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
                    pkd.y = float2_to_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
                    pkd.z = float2_to_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
                    pkd.w = float2_to_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
                    dst[q] = pkd;
                }
            }
        }
    } else if (row_ok && p.mode != USP_MODE_ACCUM) {
        // no visible key in this pass: the empty partial (0, -inf)
        uint4 *dst = reinterpret_cast<uint4 *>(orow);
        for (int q = 0; q < HD / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
    }
    if (row_ok) p.lse[grow] = lse_out;
    return true;
}

template <int HD, bool PK>
__device__ void softmax_role(const TcParams &p, uint32_t cu_s, uint32_t bar0, uint32_t tmem, uint32_t stg, int i) {
    uint32_t ns = 0, no = 0;
    for (uint32_t k = 0;; ++k) {
        uint32_t x;
        if (!unit_index(p, k, x)) break;
        const Work w = decode_work<PK>(p, cu_s, x);
        if (!softmax_unit<HD, PK>(p, cu_s, w, bar0, tmem, stg, i, ns, no)) return;
    }
}

template <int HD, bool PK>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams p) {
    using C = Cfg<HD>;
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
        // a bounded wait of an earlier CTA or launch ran out: do no work until usp_check clears it
        *skip_flag = (*reinterpret_cast<volatile int *>(p.status) != 0) ? 1u : 0u;
        for (int s = 0; s < C::kStages; ++s) {
            tc::mbar_init(bar0 + 8u * (C::K_FULL + s), 1);
            tc::mbar_init(bar0 + 8u * (C::K_EMPTY + s), 2);  // one release per MMA issuer
            tc::mbar_init(bar0 + 8u * (C::V_FULL + s), 1);
            tc::mbar_init(bar0 + 8u * (C::V_EMPTY + s), 2);
        }
        tc::mbar_init(bar0 + 8u * C::Q_FULL, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar0 + 8u * (C::S_FULL + i), 1);
            tc::mbar_init(bar0 + 8u * (C::P_FULL + i), 4);  // one arrive per softmax warp
            tc::mbar_init(bar0 + 8u * (C::O_FULL + i), 1);
        }
        tc::mbar_init(bar0 + 8u * C::DONE, 1);
        tc::mbar_init(bar0 + 8u * (C::DONE + 1), 1);
        tc::mbar_init(bar0 + 8u * C::TURN, 1);
        tc::mbar_init(bar0 + 8u * (C::TURN + 1), 1);
        tc::mbar_init(bar0 + 8u * C::Q_EMPTY, 2);  // one commit per MMA issuer
        tc::mbar_init(bar0 + 8u * C::O_EMPTY, 4);  // one arrive per softmax warp
        tc::mbar_init(bar0 + 8u * (C::O_EMPTY + 1), 4);
        tc::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
    }
    // packed samples: cu_seqlens into shared memory (when it fits), read by every role's decode
    uint32_t cu_s = 0;
    if constexpr (PK) {
        if (p.nseq + 1 <= (uint32_t)kCuCache) {
            int32_t *cs = reinterpret_cast<int32_t *>(smem + C::kCu);
            for (uint32_t e = threadIdx.x; e <= p.nseq; e += kThreads) cs[e] = p.cu[e];
            cu_s = sbase + C::kCu;
        }
    }
    if (warp == kProducerWarp && lane == 0) {
        tc::prefetch_tmap(&p.tq);
        tc::prefetch_tmap(&p.tk);
        tc::prefetch_tmap(&p.tv);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const bool skip = *skip_flag != 0;

    if (warp >= kSoftmaxWarps) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
        if (!skip) {
            if (warp == kProducerWarp && lane == 0)
                producer_role<HD, PK>(p, cu_s, sbase, bar0);
            else if (warp == kMmaWarp && lane == 0) {
                if constexpr (PK) mma_role_pk<HD, PK>(p, cu_s, sbase, bar0, tmem, 0);
                else mma_role<HD, PK>(p, cu_s, sbase, bar0, tmem, 0);
            } else if (warp == kMmaWarp1 && lane == 0) {
                if constexpr (PK) mma_role_pk<HD, PK>(p, cu_s, sbase, bar0, tmem, 1);
                else mma_role<HD, PK>(p, cu_s, sbase, bar0, tmem, 1);
            }
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        // warpgroup i: Q tile i
        if (!skip)
            softmax_role<HD, PK>(p, cu_s, bar0, tmem, sbase + (uint32_t)(C::stg_offset(PK) + warp * C::kStgSlot),
                                 warp >> 2);
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
template <int HD, bool PK>
int launch_typed(const TcParams &prm, uint32_t grid, cudaStream_t s) {
    using C = Cfg<HD>;
    // + 1024 bytes of slack for the 1024-byte alignment of the base
    constexpr int kSmem = (PK ? C::stg_offset(PK) + C::kStgBytes : C::kCu) + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return USP_ERR_CUDA;
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        // setmaxnreg.inc can only be granted from registers the launch already holds: never launch a
        // build whose register count would make the warpgroup split wait forever
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, attn_tc_kernel<HD, PK>) != cudaSuccess) return USP_ERR_CUDA;
        if ((long)fa.numRegs * kThreads < 2L * 128 * kSoftmaxRegs + 128L * kControlRegs)
            return USP_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(attn_tc_kernel<HD, PK>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
            cudaSuccess)
            return USP_ERR_CUDA;
        attr_set[dev] = true;
    }
    attn_tc_kernel<HD, PK><<<grid, kThreads, kSmem, s>>>(prm);
    return cudaGetLastError() == cudaSuccess ? USP_OK : USP_ERR_CUDA;
}

}  // namespace

int launch_attn_tc(const AttnArgs &a, cudaStream_t s) {
    const DeviceInfo *di = device_info();
    if (!di) return USP_ERR_CUDA;
    TcParams p{};
    const uint64_t q_rows = (uint64_t)a.hq * a.bs * a.L;
    // K/V rows in the head-sharded layout [rd][ud][Hkl][bs][Lr]: Hkl * ud heads of bs * L tokens
    const uint64_t kv_rows = (uint64_t)heads_per_rank(a.hkv, a.ud) * a.ud * a.bs * a.L;
    if (!make_tmap(&p.tq, a.q, q_rows, a.hd, 128) || !make_tmap(&p.tk, a.k, kv_rows, a.hd, 128) ||
        !make_tmap(&p.tv, a.v, kv_rows, a.hd, 128))
        return USP_ERR_CUDA;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse = a.lse;
    p.status = di->status;
    p.bs = (uint32_t)a.bs;
    p.rd = (uint32_t)a.rd;
    p.ud = (uint32_t)a.ud;
    p.Lr = (uint32_t)(a.L / a.rd);
    p.c = (uint32_t)(a.L / (2 * a.rd));
    p.Hl = (uint32_t)(a.hq / a.ud);
    p.Hkl = (uint32_t)heads_per_rank(a.hkv, a.ud);
    p.npairs = (p.Lr + 255) / 256;
    p.causal = a.causal;
    p.mode = a.mode;
    p.step = a.step;
    p.split = a.split;
    p.ring_rank_only = a.ring_rank_only;
    p.lpt = (p.split == USP_SPLIT_ZIGZAG && p.c % 256 == 0) ? 1 : 0;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.cu = a.cu;
    p.nseq = (uint32_t)a.nseq;
    p.L = (uint32_t)a.L;
    const uint64_t ranks = a.ring_rank_only > 0 ? 1 : (uint64_t)p.rd;
    const uint64_t units = ranks * p.ud * p.Hl * p.bs * p.npairs;
    if (units == 0) return USP_OK;
    if (units >= (1ull << 31)) return USP_ERR_UNSUPPORTED;
    p.units = (uint32_t)units;
    // unit numbering: groups of units sharing K/V (4 L hd bytes of K and V per group), in
    // super-groups of kSuperGroupKV of K/V (or one group alone of up to kSingleGroupKV) where that
    // saves DRAM traffic: not when all groups' K/V fits in the 126 MiB L2 (with a little spill), not
    // when one group's K/V alone is larger than kSingleGroupKV (not measured), and not for packed
    // samples (a unit then reads only its own sample's K/V). Working on fewer heads at a time costs
    // time of its own where the heads' K/V fits L2 anyway (measured: 7% at L = 8192 with two
    // super-groups, 50% for packed samples of 1024 with one head per super-group). Measured gains:
    // L = 131072 (32 groups of 64 MiB): DRAM reads 151 -> 60 GB per launch; with the super-groups in
    // alternating directions (decode_work) 3.6% more FLOP/s than all heads at once. L = 262144 (a head
    // group of 8 query heads: two groups of 128 MiB): 3.2% more FLOP/s, most of it from the higher
    // clock under the power cap that the smaller DRAM traffic leaves (1930 against 1810-1910 MHz).
    // One ring rank's rows alone are not grouped: under zigzag they come from two chunks whose costs
    // jump from the heaviest rows to the lightest, and a super-group numbered lightest first puts a
    // second such jump into the walk (measured at L = 262144: rank 0's rows alone 8% slower than the
    // other ranks', against 1% with all heads at once).
    p.Gl = p.Hl / p.Hkl;
    p.ngroups = p.ud * p.Hkl * p.bs;
    p.nouter = (uint32_t)ranks * p.npairs;
    const uint64_t kv_group = 4ull * (uint64_t)a.L * (uint64_t)a.hd;
    const bool grouped = !p.cu && a.ring_rank_only == 0 && (uint64_t)p.ngroups * kv_group > (160ull << 20) &&
                         kv_group <= kSingleGroupKV;
    p.sg = grouped ? (uint32_t)std::min<uint64_t>(p.ngroups, std::max<uint64_t>(1, kSuperGroupKV / kv_group))
                   : p.ngroups;
    p.sg_flip = ((p.ngroups + p.sg - 1) / p.sg - 1) & 1u;
    // persistent: one CTA per SM (the shared-memory footprint allows one), each walking its units;
    // max_ctas leaves the remaining SMs to other kernels (usp_forward_host's concurrent transfers)
    const int ctas = a.max_ctas > 0 ? std::min(a.max_ctas, di->sm_count) : di->sm_count;
    const uint32_t grid = (uint32_t)std::min<uint64_t>(units, (uint64_t)std::max(ctas, 1));
    // packed samples run a separate instantiation, so the one-sample kernel carries none of their code
    if (p.cu)
        return a.hd == 128 ? launch_typed<128, true>(p, grid, s) : launch_typed<64, true>(p, grid, s);
    return a.hd == 128 ? launch_typed<128, false>(p, grid, s) : launch_typed<64, false>(p, grid, s);
}

}  // namespace usp
