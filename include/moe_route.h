/*
 * moe_route.h -- C ABI of the GB300 (sm_103a) MoE routing library
 * (libmoe_route_gb300.so): route -> dispatch -> permute -> combine on one GPU.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers to row-major, contiguous
 *    buffers that the caller owns.  The library allocates and frees nothing,
 *    keeps no per-call state between calls and may be called from several
 *    host threads at once (each call only touches its own arguments).  Calls
 *    that may run at the same time on the GPU (other streams, other threads)
 *    must not share a dispatch workspace: it holds grid-barrier counters.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and never synchronises the host, so a sequence
 *    of calls can be captured into a CUDA graph.
 *  - Argument errors are found on the host before anything is launched; the
 *    call then returns a non-zero moe_status and launches nothing.  A failed
 *    launch returns MOE_ERR_CUDA.
 *  - Errors that only the device can see (an expert index outside [0,E), a
 *    bounded wait that ran out) are recorded in `status_word` (one int32 in
 *    device memory, may be NULL): the first error code is stored with an
 *    atomic compare-and-swap over 0, so the caller zeroes the word before the
 *    call and reads it after synchronising.  No kernel traps or asserts.
 *  - bf16 buffers are passed as `void*` (IEEE bfloat16 bit patterns).
 *  - Pointers must be 16-byte aligned; H must be a multiple of 8.
 *  - Cache use: outputs that fit in 5/8 of the GPU's L2 (the row copies,
 *    E4M3 codes and combine outputs) are stored with the default write-back
 *    policy, so that the kernel that reads them next finds them in L2; larger
 *    ones are streamed through it (evict-first).  The router leaves X in L2
 *    the same way when X fits, for the row copy that reads it again.
 *
 * Notation: N tokens, H hidden size, E experts, K experts per token,
 * slot s = n*K + k.  Limits: 1 <= E <= 256, 1 <= K <= min(E, 16),
 * N*K < 2^31, N >= 0 (N == 0 is a no-op that returns MOE_OK).
 */
#ifndef MOE_ROUTE_GB300_H
#define MOE_ROUTE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *moe_stream_t;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* a NULL required pointer, a size out of range */
    MOE_ERR_UNSUPPORTED = 2,   /* a valid request this build does not implement */
    MOE_ERR_MISALIGNED = 3,    /* a pointer not 16-byte aligned, H % 8 != 0 */
    MOE_ERR_WORKSPACE = 4,     /* workspace smaller than moe_dispatch_workspace_size() */
    MOE_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    MOE_ERR_TIMEOUT = 6,       /* (status_word only) a bounded device wait ran out */
    MOE_ERR_BAD_INDEX = 7      /* (status_word only) topk_idx entry outside [0,E) */
} moe_status;

/* Format of the E4M3 block scales (moe_dispatch_ex, moe_permute_ex). */
typedef enum moe_scale_format {
    MOE_SCALE_FP32 = 0,        /* fp32 [N*K, H/128]: the power-of-two scale s itself */
    MOE_SCALE_UE8M0 = 1        /* uint8 [N*K, H/128]: UE8M0 byte b, s = 2^(b - 127) */
} moe_scale_format;

/* Router implementation selector for moe_route_ex. */
typedef enum moe_route_algo {
    MOE_ROUTE_AUTO = 0,        /* tensor-core kernel where the shape allows it */
    MOE_ROUTE_TCGEN05 = 1,     /* tcgen05.mma + TMEM + TMA kernel (E % 8 == 0) */
    MOE_ROUTE_SIMT = 2         /* CUDA-core kernel, any E */
} moe_route_algo;

/*
 * moe_route -- the fused router.
 * Defined by the moe-engine page ("moe-engine：面向万卡集群的稀疏MoE训练基础设施"),
 * section 融合Triton路由内核: tokens @ gate_w -> softmax -> top-K -> renorm,
 * with K-round selection.  For every token n:
 *   L[e]   = sum_h X[n,h] * W_gate[h,e] (+ bias[e])    bf16 x bf16, fp32 accumulate
 *   p[e]   = softmax_e(L)[e]                          fp32
 *   idx    = the K experts with the largest logits, in descending order;
 *            equal logits go to the lower expert index; NaN counts as -inf
 *   w_k    = p[idx_k] / sum_j p[idx_j]  if renorm,  else  p[idx_k]
 * Arguments:
 *   X          bf16 [N,H]          token activations (read once)
 *   W_gate     bf16 [H,E]          gate weight, row-major ("tokens @ gate_w")
 *   bias       fp32 [E] or NULL    per-expert logit bias added before softmax
 *   topk_idx   int32 [N,K]         out: selected experts per token
 *   topk_w     fp32 [N,K]          out: routing weights
 *   status_word int32 [1] or NULL  device error word (MOE_ERR_TIMEOUT)
 * Errors: MOE_ERR_INVALID_ARG (NULL X/W_gate/outputs with N > 0, E or K out
 * of range), MOE_ERR_MISALIGNED, MOE_ERR_CUDA.
 */
MOE_API moe_status moe_route(const void *X, const void *W_gate, const float *bias,
                     int64_t N, int H, int E, int K, int renorm,
                     int32_t *topk_idx, float *topk_w, int32_t *status_word,
                     moe_stream_t stream);

/* moe_route with an explicit implementation; MOE_ERR_UNSUPPORTED if the
 * requested kernel cannot take this shape (MOE_ROUTE_TCGEN05 needs E % 8 == 0
 * and a GPU of compute capability 10.x). */
MOE_API moe_status moe_route_ex(const void *X, const void *W_gate, const float *bias,
                        int64_t N, int H, int E, int K, int renorm,
                        int32_t *topk_idx, float *topk_w, int32_t *status_word,
                        int algo, moe_stream_t stream);

/*
 * moe_route_stats -- moe_route_ex with the router statistics of the
 * moe-engine page (section 专家负载均衡) taken in the same pass:
 *   lse[n]           = log(sum_e exp(L[n,e]))   fp32 [N] or NULL: the per-token
 *                      logsumexp a z-loss squares (-inf for a token whose
 *                      logits are all -inf or NaN)
 *   expert_counts[e] = #{(n,k) : topk_idx[n,k] == e}   int32 [E] or NULL:
 *                      the expert histogram, counted in the router's epilogue
 *                      (the same values moe_dispatch writes)
 * expert_counts is overwritten (set to zero on `stream`, then accumulated by
 * the kernel).  Other arguments, layout and errors as moe_route_ex.
 */
MOE_API moe_status moe_route_stats(const void *X, const void *W_gate, const float *bias,
                           int64_t N, int H, int E, int K, int renorm,
                           int32_t *topk_idx, float *topk_w, float *lse,
                           int32_t *expert_counts, int32_t *status_word,
                           int algo, moe_stream_t stream);

/*
 * moe_load_stats -- expert-load statistics from the counts (and optionally the
 * logsumexp values) of moe_route_stats, in one small kernel:
 *   stats[0] = max_e counts[e] / mean              (imbalance ratio)
 *   stats[1] = P95(counts) / mean, P95 by linear interpolation between the
 *              sorted counts at position 0.95 * (E - 1)
 *   stats[2] = z_coef * (1/N) * sum_n lse[n]^2      (0 if lse is NULL or N == 0)
 *   stats[3] = mean = sum_e counts[e] / E
 * The ratios are 0 when every count is 0.  The sum of lse^2 is deterministic:
 * each of 1024 threads sums a fixed set of the squares in a fixed order in
 * Kahan-compensated fp32, and the 1024 per-thread sums are then added in fp64
 * in a fixed order; the count sums are exact integers.  counts int32 [E]
 * (1 <= E <= 256), lse fp32 [N] or NULL, stats fp32 [4] (all device memory).
 * Errors: MOE_ERR_INVALID_ARG (NULL counts or stats, E out of range, N < 0),
 * MOE_ERR_MISALIGNED, MOE_ERR_CUDA.
 */
MOE_API moe_status moe_load_stats(const int32_t *expert_counts, int E, const float *lse, int64_t N,
                          float z_coef, float *stats, moe_stream_t stream);

/* Bytes of device workspace moe_dispatch needs for these sizes (0 means the
 * workspace pointer may be NULL). */
MOE_API size_t moe_dispatch_workspace_size(int64_t N, int E, int K);

/*
 * moe_dispatch -- counting-sort dispatch into an expert-contiguous buffer.
 * Defined by the PithTrain page ("一万行Python构建MoE训练栈：解构4D并行、
 * DualPipeV调度与FP8算子"), §8.2 O(n) counting sort 替代 O(n log n) argsort
 * (bincount with private histograms -> prefix sum -> scatter with
 * expand_idx), specialised to one GPU (no expert-parallel ranks, no
 * all-to-all), and by the moe-engine page's conservation check
 * sum(dispatch_cnt) == N*K (section 实验结果与性能数据 / Token守恒验证).
 *   expert_counts[e]  = #{slots s : topk_idx[s] == e}
 *   expert_offsets[e] = sum_{e' < e} expert_counts[e'],  expert_offsets[E] = N*K
 *   row_map[s]        = the row of slot s in the expert-contiguous buffer;
 *                       rows are ordered by (expert, s): the stable argsort
 *                       of the slots by expert
 *   src_slot[r]       = the slot whose row is r (inverse of row_map)
 * and, when X is given, the row permute of moe_permute below.
 * Arguments:
 *   topk_idx        int32 [N,K]     expert ids (from moe_route or the caller)
 *   X               bf16 [N,H] or NULL   NULL: metadata only
 *   expert_counts   int32 [E]       out
 *   expert_offsets  int32 [E+1]     out
 *   row_map         int32 [N*K]     out
 *   src_slot        int32 [N*K] or NULL   out
 *   X_perm          bf16 [N*K,H] or NULL  out (needs X)
 *   X_fp8           uint8 [N*K,H] or NULL out, E4M3 codes (needs X, H % 128 == 0)
 *   X_scale         fp32 [N*K,H/128] or NULL  out, with X_fp8
 *   status_word     int32 [1] or NULL  device error word (MOE_ERR_BAD_INDEX)
 *   workspace       device scratch of moe_dispatch_workspace_size() bytes
 * An index outside [0,E) is reported in status_word; the outputs are then
 * unspecified but every write stays inside the buffers described above.
 * Launches: with a workspace, one cooperative launch counts, scans, scatters
 * and copies the rows; when the row copy moves 256 MiB or more (X read once
 * plus the rows written) the copy runs as a second launch of the permute
 * kernel instead.  Without a workspace: one cluster launch for the metadata,
 * then the permute kernel.
 */
MOE_API moe_status moe_dispatch(const int32_t *topk_idx, const void *X,
                        int64_t N, int H, int E, int K,
                        int32_t *expert_counts, int32_t *expert_offsets,
                        int32_t *row_map, int32_t *src_slot,
                        void *X_perm, void *X_fp8, float *X_scale,
                        int32_t *status_word,
                        void *workspace, size_t workspace_bytes,
                        moe_stream_t stream);

/*
 * moe_dispatch_ex -- moe_dispatch with a choice of block-scale format for the
 * E4M3 copy.  The PithTrain page (§7.2 架构感知的量化核, _compute_fp8_scale)
 * gives two branches of the scale rule: fp32 scales (the bit rule quoted at
 * moe_permute below) and, on Blackwell, E8M0 scales -- the same fp32 product
 * t = fl32(max(amax, 1e-4) * fl32(1/448)) converted with round-toward-+inf to
 * an unsigned 8-bit exponent (cvt.rp.satfinite.ue8m0x2.f32).  Both give the
 * same power-of-two s and hence the same E4M3 codes; MOE_SCALE_UE8M0 stores
 * one byte b per block (s = 2^(b - 127)) instead of a float.
 *   X_scale      fp32 [N*K, H/128] (MOE_SCALE_FP32, 4-byte aligned) or
 *                uint8 [N*K, H/128] (MOE_SCALE_UE8M0), with X_fp8; or NULL
 *   scale_format a moe_scale_format; anything else is MOE_ERR_INVALID_ARG
 * Every other argument, and the errors, as moe_dispatch.
 */
MOE_API moe_status moe_dispatch_ex(const int32_t *topk_idx, const void *X,
                           int64_t N, int H, int E, int K,
                           int32_t *expert_counts, int32_t *expert_offsets,
                           int32_t *row_map, int32_t *src_slot,
                           void *X_perm, void *X_fp8, void *X_scale, int scale_format,
                           int32_t *status_word,
                           void *workspace, size_t workspace_bytes,
                           moe_stream_t stream);

/*
 * moe_route_dispatch -- moe_route_ex (MOE_ROUTE_AUTO) followed by
 * moe_dispatch_ex of its own top-K ids with a bf16 row copy: the router of the
 * moe-engine page (融合Triton路由内核) and the counting sort of the PithTrain
 * page (§8.2), with the same outputs as the two calls.  Where the tensor-core
 * router runs in its split-K mode (few tokens: every CTA resident at once) the
 * whole path is ONE cooperative launch: each CTA, after its top-K epilogue,
 * counts its own slots, a bounded grid barrier follows, and every CTA then
 * forms the offsets, writes row_map for its slots and copies its tokens' rows
 * (from L2, where the router just streamed them).  Otherwise (a row copy of
 * more than 64 MiB included), or where the cooperative launch is refused, the
 * two calls run one after the other.
 *   X, W_gate, bias, renorm, topk_idx, topk_w   as moe_route
 *   expert_counts, expert_offsets, row_map, src_slot   as moe_dispatch
 *   X_perm       bf16 [N*K, H], 16-byte aligned, or NULL (metadata only)
 *   workspace    at least moe_dispatch_workspace_size(N, E, K) bytes, 256-byte
 *                aligned, zero before the first call (left zero by every call
 *                that did not time out)
 *   launches     host int or NULL: out, the number of kernels this call launched
 * Errors: those of moe_route_ex and moe_dispatch_ex; MOE_ERR_WORKSPACE when the
 * workspace is missing or too small.  The status word receives MOE_ERR_TIMEOUT
 * if the grid barrier ran out (the workspace must then be zeroed before it is
 * used again).  A split-K launch whose clusters were dropped (a profiler may run
 * a cooperative cluster launch that way) still gives the same outputs: each CTA
 * then takes the whole H range of its tile and touches no other CTA's memory.
 * The one launch is cooperative.  With the environment variable
 * MOE_FUSED_LAUNCH=noncooperative (read once per process) it is launched
 * without that attribute, for profilers that run cooperative cluster launches
 * without clusters; every CTA is then still resident at once on an otherwise
 * idle GPU (the launch is planned as one wave), but that is not guaranteed.
 */
MOE_API moe_status moe_route_dispatch(const void *X, const void *W_gate, const float *bias,
                              int64_t N, int H, int E, int K, int renorm,
                              int32_t *topk_idx, float *topk_w,
                              int32_t *expert_counts, int32_t *expert_offsets,
                              int32_t *row_map, int32_t *src_slot, void *X_perm,
                              int32_t *status_word, void *workspace, size_t workspace_bytes,
                              int *launches, moe_stream_t stream);

/*
 * moe_dispatch_ep -- expert-parallel dispatch metadata with token
 * deduplication for the tokens of one GPU: the metadata of
 * fused_dedup_prepare_dispatch on the PithTrain page (§8.2 O(n) counting sort
 * 替代 O(n log n) argsort: counts per expert and per EP rank, prefix sums,
 * send metadata, dedup scatter, counting sort, expand_idx).  The all-to-all
 * that moves the rows between GPUs is not part of this library.
 * The E experts are split over R = ep_size ranks, P = E / R consecutive
 * experts each (rank(e) = e / P).  A token is sent to a rank once, however
 * many of its K experts live there.
 *   expert_counts, expert_offsets, row_map   as moe_dispatch (int32 [E], [E+1], [N*K])
 *   rank_counts[r]    int32 [R]: tokens sent to rank r (deduplicated)
 *   rank_offsets[r]   int32 [R+1]: exclusive prefix, rank_offsets[R] = send rows
 *   send_token[row]   int32 [N*min(K,R)]: the token of send row `row`; rows are
 *                     ordered by (rank, token)
 *   slot_send_row[s]  int32 [N*K]: the send row carrying the token of slot s to
 *                     the rank of its expert
 *   expand_idx[q]     int32 [N*K]: for row q of the expert-contiguous order
 *                     (slot s), the index of s's token among its rank's send
 *                     rows: slot_send_row[s] - rank_offsets[rank(topk_idx[s])]
 *                     (what the receiving rank gathers its expert rows by)
 *   send_meta         int32 [R, P+1]: per rank, the dedup token count, then the
 *                     slot count of each of its P experts
 *   X_send            bf16 [N*min(K,R), H] or NULL: X_send[row] = X[send_token[row]]
 *                     (needs X)
 *   workspace         as moe_dispatch (moe_dispatch_workspace_size(N, E, K) bytes)
 * Three launches on `stream`.  Errors: as moe_dispatch; MOE_ERR_INVALID_ARG
 * if ep_size < 1, ep_size > E or E % ep_size != 0; MOE_ERR_UNSUPPORTED beyond
 * the one-launch dispatch's size limit (the workspace is required).  An expert
 * index outside [0,E) is reported in status_word; its slot gets no rows.
 */
MOE_API moe_status moe_dispatch_ep(const int32_t *topk_idx, const void *X,
                           int64_t N, int H, int E, int K, int ep_size,
                           int32_t *expert_counts, int32_t *expert_offsets, int32_t *row_map,
                           int32_t *rank_counts, int32_t *rank_offsets,
                           int32_t *send_token, int32_t *slot_send_row, int32_t *expand_idx,
                           int32_t *send_meta, void *X_send, int32_t *status_word,
                           void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_dispatch_noalloc -- moe_dispatch without a caller-provided workspace.
 * The pages have no counterpart: this is a convenience of this library for
 * callers that cannot allocate device memory when they dispatch -- engines that
 * fix their whole device-memory plan up front and forbid later allocation,
 * code running where cudaMalloc would block or synchronise the device, or C
 * callers with no device allocator of their own.  The inputs and outputs are
 * still the caller's (same meaning as in moe_dispatch); the scratch is a
 * 1 MiB + 256 B array compiled into the library, which every GPU that loads
 * the library holds until the process exits.  The call allocates and frees
 * nothing.
 *  - The first call on each device looks up the array's device address
 *    (with that device current) and caches it; make that first call before
 *    any stream capture.
 *  - Every call clears the array's barrier counters on `stream` and then uses
 *    the whole array: calls that may overlap on the GPU (other streams, other
 *    host threads) race on it and must be serialised by the caller.
 *  - Limit: the launch takes C = min(N, number of SMs) CTAs, each with
 *    ceil(N / C) tokens, and a CTA holds at most 16384 slots, so the call
 *    needs ceil(N / C) * K <= 16384 (on a 152-SM GB300 with K = 3: up to
 *    N = 830072); larger calls return MOE_ERR_UNSUPPORTED and launch nothing.
 *  - Every argument check of moe_dispatch runs on the host before any CUDA
 *    call: a rejected call queues nothing on `stream`.
 */
MOE_API moe_status moe_dispatch_noalloc(const int32_t *topk_idx, const void *X,
                                int64_t N, int H, int E, int K,
                                int32_t *expert_counts, int32_t *expert_offsets,
                                int32_t *row_map, int32_t *src_slot,
                                void *X_perm, void *X_fp8, float *X_scale,
                                int32_t *status_word, moe_stream_t stream);

/*
 * moe_permute -- the row permute of the dispatch, on its own.
 * The gathered_tokens input of forward_mlp on the PithTrain page
 * (§6.1 模型协议先行): X_perm[row_map[n*K+k], :] = X[n, :].
 * With X_fp8/X_scale (H % 128 == 0) every 1x128 block of X[n,:] is also
 * quantised with the power-of-two scale of §7.2 架构感知的量化核
 * (_compute_fp8_scale, fp32-scale branch):
 *   s = pow2ceil(fl32(max(amax, 1e-4) * fl32(1/448))),  q = E4M3_rn_satfinite(x / s)
 * and q, s are written for every destination row of the token.
 * row_map must be a permutation of [0, N*K) (as moe_dispatch writes it);
 * rows outside [0, N*K) are skipped and reported as MOE_ERR_BAD_INDEX.
 * X_perm may be NULL when only the E4M3 copy is wanted.
 */
MOE_API moe_status moe_permute(const void *X, const int32_t *row_map,
                       int64_t N, int H, int K,
                       void *X_perm, void *X_fp8, float *X_scale,
                       int32_t *status_word, moe_stream_t stream);

/* moe_permute with a choice of block-scale format (see moe_dispatch_ex). */
MOE_API moe_status moe_permute_ex(const void *X, const int32_t *row_map,
                          int64_t N, int H, int K,
                          void *X_perm, void *X_fp8, void *X_scale, int scale_format,
                          int32_t *status_word, moe_stream_t stream);

/*
 * moe_combine -- weighted gather back to token order.
 * The weighted part of forward_aggregate on the PithTrain page (§6.1
 * 模型协议先行, "weighted expert output"):
 *   out[n,:] = sum_{k=0}^{K-1} topk_w[n,k] * Y[row_map[n*K+k], :]
 * accumulated in fp32 in k order and rounded to bf16 (nearest even).
 * Arguments: Y bf16 [N*K,H] (expert outputs in the expert-contiguous order),
 * row_map int32 [N*K], topk_w fp32 [N,K], out bf16 [N,H].
 * Rows outside [0, N*K) contribute nothing and are reported as
 * MOE_ERR_BAD_INDEX in status_word.
 */
MOE_API moe_status moe_combine(const void *Y, const int32_t *row_map, const float *topk_w,
                       int64_t N, int H, int K, void *out,
                       int32_t *status_word, moe_stream_t stream);

/*
 * moe_combine_residual -- moe_combine plus the residual connection: the whole
 * of forward_aggregate on the PithTrain page (§6.1 模型协议先行, "weighted
 * expert output + residual connection"), fused into the same pass:
 *   out[n,:] = sum_{k=0}^{K-1} topk_w[n,k] * Y[row_map[n*K+k], :] + residual[n,:]
 * with the weighted sum accumulated in fp32 in k order, the residual added in
 * fp32, and one rounding to bf16 (nearest even).
 * Arguments: as moe_combine, plus residual bf16 [N,H] (required, 16-byte
 * aligned).  out may be the residual buffer itself (in-place update of the
 * residual stream); any other overlap of out with Y or residual is undefined.
 * Errors: as moe_combine; a NULL residual with N > 0 is MOE_ERR_INVALID_ARG.
 */
MOE_API moe_status moe_combine_residual(const void *Y, const int32_t *row_map, const float *topk_w,
                                const void *residual, int64_t N, int H, int K, void *out,
                                int32_t *status_word, moe_stream_t stream);

/* A static, human-readable name for a status code. */
MOE_API const char *moe_status_string(moe_status status);

/* ABI version of this header (bumped on any signature change). */
MOE_API int moe_abi_version(void);
#define MOE_ABI_VERSION 1

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_GB300_H */
