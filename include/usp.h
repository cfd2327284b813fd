/*
 * usp.h -- C ABI of the USP-Attention forward hot path on one GPU (sm_103a).
 *
 * USP-Attention ("USP: 统一序列并行方法用于长上下文生成式AI", section 三, Algorithm 1) runs
 * AllToAll4D over a Ulysses group, ring attention with log-sum-exp merging over a Ring group, and the
 * inverse AllToAll4D. Here the ud x rd process grid is a set of VIRTUAL ranks inside one device:
 * every "rank" is an index range of one device buffer, the all-to-all is an on-device permute, and
 * the ring's point-to-point sends become the order in which KV blocks are fed to the attention
 * kernel. No call communicates between devices.
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers unless stated otherwise. The caller owns every buffer; the
 *    library never allocates caller-visible memory and never frees anything.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream). Argument
 *    errors are returned before anything is launched. USP_ERR_CUDA reports a launch failure.
 *  - Device-side waits inside kernels are bounded; a wait that runs out sets a per-device status word
 *    and the kernel returns early. usp_check() synchronises the stream and reports it as
 *    USP_ERR_TIMEOUT.
 *  - Virtual rank (u, r) (Ulysses rank u, ring rank r) has flat id vr = r * ud + u (ring-major; the
 *    USP review's Tip 7 orders process groups TP -> Ulysses -> Ring from low to high).
 *  - Notation: c = L / (2 rd) zigzag chunk length, Lr = L / rd ring-local length,
 *    Lu = L / (rd ud) tokens per virtual rank, Hl = H / ud heads per Ulysses rank.
 *  - Shapes: L % (2 rd) == 0 and Lr % ud == 0 (equal chunks, as torch.chunk gives in the pages'
 *    setting); H % ud == 0 for an all-to-all (the Ulysses degree divides the head count, the
 *    Context-Parallel page's "head 数整除检查"); hq % hkv == 0. One exception: the forward
 *    all-to-all of K/V also accepts fewer heads than Ulysses ranks when H divides ud (GQA/MQA,
 *    below). Violations return USP_ERR_SHAPE.
 *  - GQA/MQA with hkv < ud: the USP review's section 三 gives AllToAll4D the job of handling K/V
 *    head counts that differ from Q's, without details. Reading taken here: Ulysses rank u' holds
 *    query heads [u' Hl, (u' + 1) Hl), which all read KV head u' / (ud / hkv); the forward
 *    all-to-all sends it that head only, so each KV head is replicated on ud / hkv ranks and the
 *    head-sharded K/V carries Hkl = 1 head per rank (Hkl = hkv / ud otherwise).
 *  - Sizes: every row count handled by one call must stay below 2^31.
 */
#ifndef USP_H
#define USP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define USP_API __attribute__((visibility("default")))
#else
#define USP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *usp_stream_t; /* identical to cudaStream_t */

typedef enum {
    USP_OK = 0,
    USP_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad enum value */
    USP_ERR_SHAPE = -2,       /* divisibility rules above */
    USP_ERR_DTYPE = -3,       /* unknown dtype code */
    USP_ERR_ALIGN = -4,       /* a pointer is not aligned as the call requires */
    USP_ERR_UNSUPPORTED = -5, /* valid but not implemented (e.g. head_dim not 64/128) */
    USP_ERR_CUDA = -6,        /* a CUDA runtime call or launch failed */
    USP_ERR_TIMEOUT = -7      /* a bounded device-side wait ran out (reported by usp_check) */
} usp_status;

typedef enum { USP_F32 = 0, USP_BF16 = 1 } usp_dtype;

/* How the global sequence is divided among the ring ranks (ring-local row p of ring rank r holds
 * global token pos(r, p); every split keeps pos increasing in p). */
typedef enum {
    USP_SPLIT_ZIGZAG = 0, /* Algorithm 2: chunks r and 2 rd - 1 - r of 2 rd equal chunks (load-balanced) */
    USP_SPLIT_BASIC = 1,  /* the plain ring: tokens [r L/rd, (r+1) L/rd) (USP review, "basic-ring") */
    USP_SPLIT_STRIPE = 2  /* Striped Attention's round robin: tokens r, r + rd, r + 2 rd, ... */
} usp_split;

/* Shape of one tensor moved by a permute. */
typedef struct {
    int64_t bs;      /* batch size */
    int64_t L;       /* global sequence length */
    int32_t H;       /* heads moved by this call */
    int32_t hd;      /* elements per row: the head dim (1 for an lse tensor) */
    int32_t dtype;   /* usp_dtype: element size 4 (USP_F32) or 2 (USP_BF16) */
    int32_t rd;      /* ring degree  >= 1 */
    int32_t ud;      /* Ulysses degree >= 1 */
    int32_t H_total; /* heads per token in the natural / sequence-sharded tensor (0 means H) */
    int32_t h0;      /* first head of the window [h0, h0 + H) in that tensor */
    int32_t split;   /* usp_split; USP_SPLIT_ZIGZAG (0) unless stated */
} usp_dims;

/*
 * usp_extract_local -- the zigzag load-balanced split (step a1).
 * Source: USP review, section 三, Algorithm 2 (seq.chunk(2 rd); rank r keeps chunks r and
 * 2 rd - r - 1; then the u-th of ud equal parts); Context-Parallel page, Fig. 2.
 *
 *   natural  : (bs, L, H_total, hd) row-major, natural token order; the call reads/writes the heads
 *              [h0, h0 + H) of it.
 *   local    : [rd][ud][bs][Lu][H][hd] (all virtual ranks, vr-major), or (bs, Lu, H, hd) for one rank.
 *   Local slot (r, u, b, j, h) holds token zig(r, u Lu + j) of head h0 + h, where
 *   zig(r, p) = r c + p for p < c and (2 rd - 1 - r) c + (p - c) otherwise (d.split selects the basic
 *   or stripe split instead: pos(r, p) = r Lr + p or p rd + r).
 *
 * inverse == 0: src = natural, dst = local.  inverse != 0: src = local, dst = natural (restores
 * natural order; heads outside the window are left untouched).
 * vr == -1: all ud * rd virtual ranks in one launch; 0 <= vr < ud * rd: only that rank's part.
 * Bit-exact copy. Both pointers must be 16-byte aligned when hd * elem_size is a multiple of 16,
 * else 4-byte aligned. src and dst must not overlap.
 */
USP_API int usp_extract_local(const void *src, void *dst, usp_dims d, int vr, int inverse, usp_stream_t stream);

/*
 * usp_a2a4d -- AllToAll4D inside every Ulysses group (steps a2 and a5).
 * Source: USP review, section 三 (AllToAll4D: Q, K, V of shape (bs, L/N, hc, hd) become
 * (hc/N, bs, L, hd); Algorithm 1 steps 1-3, and step 5 with scatter/gather indices swapped).
 *
 *   sequence-sharded : [rd][ud][bs][Lu][H_total][hd], heads [h0, h0 + H) taking part.
 *   head-sharded     : [rd][ud][Hl][bs][Lr][hd] (compact, Hl = H / ud).
 *   head-sharded[r][u'][h'][b][u Lu + j] = sequence-sharded[r][u][b][j][h0 + u' Hl + h'],
 *   i.e. pieces are gathered by source Ulysses rank ascending.
 * dir == +1: sequence-sharded -> head-sharded.  dir == -1: head-sharded -> sequence-sharded.
 * dir == +1 with H < ud and ud % H == 0 replicates (K/V under GQA/MQA): head-sharded is
 *   [rd][ud][1][bs][Lr][hd] and head-sharded[r][u'][0][b][u Lu + j] =
 *   sequence-sharded[r][u][b][j][h0 + u' / (ud / H)]. dir == -1 with H < ud is the adjoint of that:
 *   each head receives the SUM of its ud / H replicas (fp32 sum, rounded once), which is what the
 *   gradients of replicated K/V need.
 * Alignment and overlap rules as for usp_extract_local. An lse tensor is moved with hd = 1, USP_F32.
 */
USP_API int usp_a2a4d(const void *src, void *dst, usp_dims d, int dir, usp_stream_t stream);

/*
 * usp_a2a4d_multi -- usp_a2a4d for up to four tensors in one launch (e.g. step a5 of out and lse
 * together). Source: as usp_a2a4d.
 *
 *   n         : number of tensors, 1 <= n <= 4
 *   src, dst  : HOST arrays of n DEVICE pointers, each pair as src / dst of usp_a2a4d.
 *   d         : HOST array of n dims; bs, L, rd and ud must agree (USP_ERR_SHAPE otherwise); H,
 *               H_total, h0, hd and dtype may differ (out rows of hd elements with lse rows, hd = 1).
 *   dir       : +1 or -1 for every tensor, as usp_a2a4d.
 * Bit-exactly the result of one usp_a2a4d call per tensor. Alignment and overlap rules as for
 * usp_extract_local, per tensor.
 */
USP_API int usp_a2a4d_multi(int n, const void *const *src, void *const *dst, const usp_dims *d, int dir,
                            usp_stream_t stream);

/*
 * usp_extract_a2a -- the zigzag split followed by AllToAll4D (steps a1 + a2) in one pass, for up to
 * four tensors (e.g. Q, K and V, or out and lse) in one launch; inverse != 0 runs AllToAll4D's
 * inverse followed by the inverse split (a5 + a7).
 * Source: USP review, Algorithm 2 and section 三 (AllToAll4D). Composing the two maps gives
 *   head-sharded[r][u'][h'][b][p] = natural[b][zig(r, p)][h0 + u' Hl + h'],
 * i.e. row p of ring rank r is global token zig(r, p) (the all-to-all gathers the Ulysses ranks'
 * pieces in rank order, which restores Algorithm 2's ring-local sequence). Bit-exactly the result of
 * usp_extract_local (vr = -1) then usp_a2a4d (dir = +1), with one read and one write per tensor.
 *
 *   n         : number of tensors, 1 <= n <= 4
 *   src, dst  : HOST arrays of n DEVICE pointers. inverse == 0: src[k] natural (bs, L, H_total, hd),
 *               dst[k] head-sharded [rd][ud][H/ud][bs][Lr][hd] (or, when H < ud and ud % H == 0,
 *               [rd][ud][1][bs][Lr][hd] holding head u' / (ud / H) on rank u', as usp_a2a4d);
 *               inverse != 0: the other way round (with H < ud, the sum of each head's replicas,
 *               as usp_a2a4d dir = -1); heads outside the window of the natural tensor are left
 *               untouched.
 *   d         : HOST array of n dims; bs, L, rd, ud and split must agree (USP_ERR_SHAPE
 *               otherwise); H, H_total and h0 may differ (Q and K/V head counts under GQA), and so
 *               may hd and dtype (out rows of hd elements with lse rows of one fp32, hd = 1).
 * Alignment and overlap rules as for usp_extract_local.
 */
USP_API int usp_extract_a2a(int n, const void *const *src, void *const *dst, const usp_dims *d, int inverse,
                            usp_stream_t stream);

/* Attention modes (step a3 with the merge of step a4). */
typedef enum {
    USP_MODE_FUSED = 0, /* the whole ring: every ring step folded into one online softmax */
    USP_MODE_STEP = 1,  /* one ring step `step`: write its partial (o_t, lse_t); empty rows get
                           o = 0, lse = -inf */
    USP_MODE_ACCUM = 2  /* one ring step `step`, merged into the (out, lse) already in the buffers */
} usp_mode;

typedef struct {
    int64_t bs;     /* batch size */
    int64_t L;      /* global sequence length */
    int32_t hq;     /* query heads (global, of this head group) */
    int32_t hkv;    /* KV heads (global, of this head group); GQA: q head h reads KV head h / (hq/hkv) */
    int32_t hd;     /* head dim: 64 or 128 */
    int32_t rd;     /* ring degree */
    int32_t ud;     /* Ulysses degree */
    int32_t dtype;  /* usp_dtype of q, k, v and out */
    int32_t causal; /* nonzero: key at global position j visible to query at i iff j <= i */
    float scale;    /* softmax scale; <= 0 means 1/sqrt(hd) */
    int32_t mode;   /* usp_mode */
    int32_t step;   /* ring step t for USP_MODE_STEP / USP_MODE_ACCUM, 0 <= t < rd */
    int32_t split;  /* usp_split of q / k / v (must match the split the permutes used) */
    int32_t ring_rank_only; /* 0: every ring rank; k > 0: only ring rank k - 1's query rows are
                               computed and written (its share of the work, e.g. to time one rank) */
    int32_t nseq;   /* packed samples: 0 (or 1) = one sequence; n > 1 = n samples concatenated */
    const int32_t *cu_seqlens; /* DEVICE array of nseq + 1 cumulative sample lengths, 0 = cu[0] <
                               cu[1] < ... < cu[nseq] = L (the same packing for every batch element);
                               a query sees only keys of its own sample. Read by the kernels only;
                               values that break these rules give meaningless masks, not faults. */
} usp_attn_desc;

/*
 * usp_attn_fwd -- LoadBalance-RingAttention forward over all virtual ring ranks (steps a3 + a4).
 * Source: USP review, Algorithm 1 step 4; Context-Parallel page, section 先弄清楚 (each KV block
 * gives o_j and lse_j; lse = log(e^lse1 + e^lse2), o = e^(lse1-lse) o1 + e^(lse2-lse) o2) and Fig. 1
 * (at step t ring rank r works on the KV block of rank (r - t) mod rd).
 *
 *   q, out : [rd][ud][hq/ud][bs][Lr][hd]   (head-sharded, as usp_a2a4d dir=+1 writes it)
 *   k, v   : [rd][ud][Hkl][bs][Lr][hd], Hkl = hkv/ud, or 1 when hkv < ud (ud % hkv == 0; each
 *            Ulysses rank holds the replica of KV head u' / (ud / hkv), as usp_a2a4d writes it)
 *   lse    : [rd][ud][hq/ud][bs][Lr] fp32, natural log of the row's softmax normaliser.
 * Row p of ring rank r is the token at global position zig(r, p); the causal mask compares global
 * positions. Packed samples (d.nseq > 1; the sequence packing of the Context-Parallel page's
 * ByteScale section): the split is that of the packed sequence, and a query sees only keys of its
 * own sample, so tiles across sample boundaries are skipped. Scores are scale * <q, k>; inputs bf16 (tensor cores, fp32 accumulation, bf16 out) or
 * fp32 (fp32 arithmetic, fp32 out). All pointers 16-byte aligned. out/lse must not overlap inputs.
 * In USP_MODE_ACCUM, out and lse are read and rewritten in place.
 */
USP_API int usp_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, usp_attn_desc d,
                 usp_stream_t stream);

/*
 * usp_lse_merge -- fold one partial into a running one, in place (step a4 as a standalone pass).
 * Source: Context-Parallel page, section 先弄清楚 (the online-softmax merge equation).
 *   (o_acc, lse_acc) <- (e^(l1 - l) o_acc + e^(l2 - l) o_new, l),  l = log(e^l1 + e^l2),
 *   l1 = lse_acc, l2 = lse_new. lse = -inf marks an empty partial (weight 0); two empty partials
 *   give (0, -inf).
 *   o_acc, o_new : rows x hd of `dtype` (row-major);  lse_acc, lse_new : rows fp32.
 * Pointers 16-byte aligned; hd * elem_size a multiple of 16. fp32 arithmetic.
 */
USP_API int usp_lse_merge(void *o_acc, float *lse_acc, const void *o_new, const float *lse_new, int64_t rows,
                  int32_t hd, int32_t dtype, usp_stream_t stream);

/*
 * usp_forward -- the whole USP-Attention forward on device buffers: for every head group, the split
 * and AllToAll4D of Q, K, V (usp_extract_a2a), the ring attention (usp_attn_fwd, USP_MODE_FUSED) and
 * the inverse AllToAll4D + inverse split of out and lse back to natural order.
 * Source: USP review, Algorithm 1 (steps 1-5) and Algorithm 2; the head groups follow the UPipe
 * page's headwise chunking (the result does not depend on the grouping).
 *
 *   q                : (bs, L, hq, hd) natural order;  k, v : (bs, L, hkv, hd)
 *   out              : (bs, L, hq, hd) natural order;  lse  : (bs, L, hq) fp32, natural log
 *   d                : as for usp_attn_fwd; d.mode must be USP_MODE_FUSED
 *   head_chunk       : query heads per group (0 = all); must divide hq and be a multiple of hq/hkv;
 *                      the group's query head count must divide by ud and its KV head count
 *                      divide by ud or divide ud (replicated K/V)
 *   workspace        : DEVICE buffer, 256-byte aligned, at least usp_forward_workspace_size(d,
 *                      head_chunk, 0) bytes; owned by the caller, clobbered by the call
 * Asynchronous on `stream`; calls that share a workspace must be ordered on one stream.
 */
USP_API int usp_forward(const void *q, const void *k, const void *v, void *out, float *lse, usp_attn_desc d,
                        int head_chunk, void *workspace, size_t workspace_bytes, usp_stream_t stream);

/*
 * usp_forward_host -- usp_forward from HOST input buffers to HOST output buffers (same layouts).
 * Two paths, chosen per call:
 *   direct -- when all five host buffers are page-locked and mapped into the current device's address
 *     space (cudaHostAlloc, cudaHostRegister, a pinned torch tensor: cudaPointerGetAttributes reports
 *     cudaMemoryTypeHost with a device pointer), the kernels read q, k, v and write out and lse in host
 *     memory themselves over the CPU-GPU link. The head groups alternate between two slots of device
 *     buffers in the workspace: group g's attention runs on `stream` while group g+1's split +
 *     all-to-all gathers from host memory and group g-1's inverse scatters to host memory on two
 *     library streams. For bf16 without packed samples, each transfer gets a few thread blocks,
 *     enough to finish within about half of an attention, and the attention leaves that many SMs
 *     free; the first gather and the last scatter run on the whole GPU. Each buffer must lie within
 *     one page-locked allocation.
 *   copy -- otherwise, pipelined per head group: the host-to-device copy of group g+1 and the
 *     device-to-host copy of group g-1 overlap the kernels of group g, on three streams the library
 *     keeps per device; pageable buffers work but their copies do not overlap.
 * Either way the whole call is ordered after earlier work on `stream`, and later work on `stream`
 * waits for it (the host outputs are complete once `stream` is synchronised); calls on one device
 * are serialised by the library (its streams are per device).
 *   workspace : DEVICE buffer of at least usp_forward_workspace_size(d, head_chunk, 1) bytes
 *               (copy path: two staging slots per direction plus the full lse; direct path: two
 *               slots of the head-sharded buffers), 256-byte aligned.
 * Calls on one device are serialised on the library's streams; calls that share a workspace must be
 * ordered on one stream.
 */
USP_API int usp_forward_host(const void *q_host, const void *k_host, const void *v_host, void *out_host,
                             float *lse_host, usp_attn_desc d, int head_chunk, void *workspace,
                             size_t workspace_bytes, usp_stream_t stream);

/* Bytes of workspace usp_forward (host_buffers == 0) or usp_forward_host (host_buffers != 0) needs;
 * 0 if the arguments are invalid. */
USP_API size_t usp_forward_workspace_size(usp_attn_desc d, int head_chunk, int host_buffers);

/* Size of the library-owned scratch array used by usp_forward_noalloc (32 MiB). */
#define USP_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * usp_forward_noalloc -- usp_forward without a caller workspace; this entry point allocates nothing.
 * The pages have no counterpart: it exists for callers that cannot hand out device memory, e.g. a
 * plugin inside an application whose memory manager owns all device memory and forbids allocations
 * outside its pool, or a caller on a latency-critical path that must not call cudaMalloc / cudaFree
 * (they can synchronise the device). The workspace is a fixed array of USP_NOALLOC_SCRATCH_BYTES
 * that this library places on every GPU that loads it, kept until the process exits.
 *   Arguments, layouts and shape rules as for usp_forward. Shapes whose workspace
 *   (usp_forward_workspace_size(d, head_chunk, 0)) exceeds USP_NOALLOC_SCRATCH_BYTES return
 *   USP_ERR_UNSUPPORTED before anything runs: choose a smaller head_chunk (e.g. L = 8192, hd = 128,
 *   bf16 fits with 2 query heads per group for MHA).
 *   The device is the CURRENT device (cudaGetDevice): q, k, v, out, lse and the stream must belong to
 *   it, since the array used is the current device's copy.
 *   The first call on a device looks up the array's device address (once per device, cached); make
 *   that first call before any stream capture begins. The cached address is not refreshed: after a
 *   cudaDeviceReset of that device (which unloads the library's module there), do not call this
 *   entry point again in the same process.
 *   Every call on a device uses the same array, and calls that overlap on the GPU race on it (e.g.
 *   two streams at once): order them on one stream. The array keeps the last call's contents; the
 *   call writes every workspace byte it reads, so nothing needs to start at zero.
 */
USP_API int usp_forward_noalloc(const void *q, const void *k, const void *v, void *out, float *lse, usp_attn_desc d,
                                int head_chunk, usp_stream_t stream);

/*
 * usp_attn_bwd_delta -- D_i = <dout_i, out_i> for every row (the softmax backward's row term).
 * Source: the gradient of softmax attention (UPipe page, attention formula; the backward needs the
 * forward's inputs and output): with P = softmax(S), dS = P o (dP - D) and D_i = sum_j P_ij dP_ij,
 * which equals <dout_i, out_i> because out_i = sum_j P_ij v_j and dP_ij = <dout_i, v_j>.
 *   out, dout : rows x hd of `dtype`, row-major, any layout whose rows are contiguous (natural or
 *               head-sharded);  delta : rows fp32 (same row order). fp32 accumulation.
 * Pointers 16-byte aligned; hd * elem_size a multiple of 16.
 */
USP_API int usp_attn_bwd_delta(const void *out, const void *dout, float *delta, int64_t rows, int32_t hd,
                               int32_t dtype, usp_stream_t stream);

/*
 * usp_attn_bwd -- backward of usp_attn_fwd (the whole ring, USP_MODE_FUSED) over all virtual ring
 * ranks: the gradients of out with respect to q, k and v.
 * Source: the YunChang page runs its hybrid zigzag test with the backward (--use_bwd); the
 * Context-Parallel page pairs the forward's gather of K/V with a reduce-scatter of their gradients
 * in the backward; the formulas are the chain rule through softmax (usp_attn_bwd_delta):
 *   P_ij = exp(s_ij - lse_i), dP_ij = <dout_i, v_j>, dS_ij = P_ij (dP_ij - D_i),
 *   dq_i = scale sum_j dS_ij k_j, dk_j = scale sum_i dS_ij q_i, dv_j = sum_i P_ij dout_i,
 * over the same causal (query, key) pairs as the forward. In a multi-GPU ring, the dk/dv partials of
 * a KV block travel with it and are home after rd steps; here each KV block's gradient is formed in
 * place.
 *   q, dout, dq : [rd][ud][hq/ud][bs][Lr][hd]   (head-sharded)
 *   k, v, dk, dv: [rd][ud][Hkl][bs][Lr][hd]     (Hkl as for usp_attn_fwd; with replicated K/V each
 *                 replica receives the gradient from its own rank's query heads only, and the
 *                 replica sum happens in the inverse all-to-all, usp_a2a4d dir = -1)
 *   lse, delta  : [rd][ud][hq/ud][bs][Lr] fp32: the forward's lse and usp_attn_bwd_delta's output
 * d as for usp_attn_fwd with d.mode == USP_MODE_FUSED and d.ring_rank_only == 0. All pointers
 * 16-byte aligned; outputs must not overlap inputs. Arithmetic in fp32; gradients written in the
 * input dtype.
 */
USP_API int usp_attn_bwd(const void *q, const void *k, const void *v, const void *dout, const float *lse,
                         const float *delta, void *dq, void *dk, void *dv, usp_attn_desc d, usp_stream_t stream);

/*
 * usp_backward -- the whole USP-Attention backward on device buffers, the counterpart of
 * usp_forward: D from out and dout, then for every head group the split and AllToAll4D of q, k, v,
 * dout, lse and D, the ring backward (usp_attn_bwd), and the inverse AllToAll4D (summing replicas of
 * replicated K/V) and inverse split of dq, dk, dv back to natural order.
 * Source: as usp_forward and usp_attn_bwd; the UPipe page's headwise chunks each take their own
 * gradients, so the grouping does not change the result.
 *   q, out, dout, dq : (bs, L, hq, hd) natural order;  k, v, dk, dv : (bs, L, hkv, hd)
 *   lse              : (bs, L, hq) fp32, the forward's
 *   d, head_chunk    : as for usp_forward
 *   workspace        : DEVICE buffer, 256-byte aligned, at least usp_backward_workspace_size(d,
 *                      head_chunk) bytes; owned by the caller, clobbered by the call
 */
USP_API int usp_backward(const void *q, const void *k, const void *v, const void *out, const float *lse,
                         const void *dout, void *dq, void *dk, void *dv, usp_attn_desc d, int head_chunk,
                         void *workspace, size_t workspace_bytes, usp_stream_t stream);

/* Bytes of workspace usp_backward needs; 0 if the arguments are invalid. */
USP_API size_t usp_backward_workspace_size(usp_attn_desc d, int head_chunk);

/* Synchronise `stream`, then report (and clear) the device status word of the current device:
 * USP_OK, USP_ERR_TIMEOUT, or USP_ERR_CUDA if the synchronisation itself failed. */
USP_API int usp_check(usp_stream_t stream);

/*
 * usp_selftest_timeout -- exercises the failure path of the bounded device-side waits without a
 * fault: one CTA waits, through the same bounded mbarrier wait every kernel of this library uses, on
 * a barrier nothing ever arrives on, for at most limit_us microseconds. The wait runs out, the kernel
 * records USP_ERR_TIMEOUT in the device status word and returns; the context stays usable.
 * usp_check then reports USP_ERR_TIMEOUT and clears the word; the tensor-core (bf16) attention
 * kernels, the ones with device-side waits, do no work when launched while the word is set
 * (usp_check reports the timeout for them too).
 *   limit_us : 1 .. 1000000, else USP_ERR_INVALID_ARG.
 */
USP_API int usp_selftest_timeout(int64_t limit_us, usp_stream_t stream);

/* Static, human-readable text for a status code. */
USP_API const char *usp_strerror(int status);

/* ABI version: (major << 16) | minor. */
USP_API int usp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* USP_H */
