// route_tc.cu -- the fused router on the 5th-generation tensor cores.
//
// Method (moe-engine page, "moe-engine：面向万卡集群的稀疏MoE训练基础设施",
// section 融合Triton路由内核): logits = tokens @ gate_w, softmax over E,
// top-K, renorm -- in one pass over X, so the logits never reach HBM.
//
// GB300 design (not the page's 64x64 SRAM tiling).  One CTA per SM, 10 warps:
//   warp 0     TMA producer: X tile [128 x 64] and gate-weight slab [64 x EP]
//              per K-step, 128-byte swizzle, into a ring of `stages` shared
//              memory slots (full/empty mbarrier pairs), running ahead across
//              tile boundaries;
//   warp 1     MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16 -> fp32), M = 128,
//              N = E rounded up to 16, four K = 16 steps per slot, into one of
//              two TMEM accumulators (128 lanes x N fp32 columns each);
//   warps 2-9  epilogue: two warps per TMEM lane quarter, each taking half of
//              the expert columns of its 32 tokens.
// X is K-major (row-major [N,H]); the gate weight [H,E] is read as stored, as an
// MN-major B operand (E contiguous), so no transpose pass is needed.
//
// Two modes:
//   * persistent (many tokens): CTA c takes tiles c, c + grid, ...; the
//     epilogue of tile t overlaps the MMAs of tile t + 1 (double-buffered TMEM).
//   * split (few tokens: the 128-token tiles alone would leave most SMs idle):
//     a thread-block cluster of S CTAs shares a tile, CTA r taking 1/S of the
//     H range; the partial logits go through distributed shared memory to the
//     CTA that owns those 128/S tokens, which sums the S slices in a fixed order
//     and finishes its tokens with 2S threads per token.
// Top-K: each thread keeps sorted top-K lists in registers (a candidate enters
// with K compare-exchange steps, lists fed with increasing expert ids so equal
// logits keep the lower id first); the lists of a token are merged by K rounds
// of "take the best head" -- K-round selection over list heads, through shared
// memory between the two column halves or warp shuffles between the threads of
// a token.  Ties go to the lower expert index; NaN counts as -inf.
//
// The epilogue is written as rolled loops: it runs once or a few times per CTA,
// and straight-line unrolled code there is dominated by instruction fetch.
//
// Every mbarrier wait is bounded (2 s of %globaltimer); on expiry the CTA records
// MOE_ERR_TIMEOUT, drains its outstanding copies and MMAs, still reaches the
// cluster barriers (so no peer waits forever), frees TMEM and exits.
#include <math.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;                       // tokens per tile (UMMA M)
constexpr int kBK = 64;                        // bf16 per 128-byte swizzle row (one K-step)
constexpr int kEpiWarps = 8;                   // split mode (and the dispatch tail fused into it)
constexpr int kThreads = 64 + 32 * kEpiWarps;  // 320
constexpr int kWarps = kThreads / 32;

// Epilogue width per mode: 8 warps, two per TMEM lane quarter, so each token's
// columns are split into two parts in persistent mode.  (The persistent
// epilogue is written for 2 or 4 parts; 16 warps with four parts measured no
// faster on GB300 at E = 128, K = 8: the candidate loop is bound by its
// instruction count, not by latency, and the extra merge level cost more than
// the shorter scans saved.)
template <int KMAX, bool SPLIT>
struct TcShape {
    static constexpr int kEpi = kEpiWarps;
    static constexpr int kThr = 64 + 32 * kEpi;
    static constexpr int kParts = kEpi / 4;       // column parts per token (persistent mode)
};
// rows of the per-CTA count table in the dispatch workspace: the same bound as the
// dispatch kernel's table (dispatch.cu), which sizes moe_dispatch_workspace_size()
constexpr int kFuseMaxCtas = 1024;
constexpr int64_t kFuseMaxCopyBytes = 64ll << 20;   // fused row copies up to this size
constexpr uint32_t kABytes = kBM * kBK * 2;    // 16 KiB X tile per slot
constexpr uint32_t kBBoxBytes = kBK * 64 * 2;  // 8 KiB per 64-expert gate box
constexpr int kMaxStages = 12;
constexpr int kEmpty = 0x7fffffff;             // index of an empty list slot

struct TcSmemTail {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

struct TcParams {
    const float *bias;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *status;
    float *lse;            // [N] per-token logsumexp of the logits, or nullptr
    int32_t *counts;       // [E] slot count per expert (accumulated; zeroed by the caller), or nullptr
    int N, H, E, K, renorm;
    int need_z;            // the full softmax denominator is needed (renorm off, or lse requested)
    int EP, NP, stages, nsplit, kb_per, tiles;
    int tile_rows;         // tokens per tile (kBM, or fewer so that the tiles fill whole waves of SMs)
    int kpack;             // persistent mode: K-steps per ring stage (1, or 2 with the 3D X map)
    int x_keep;            // X fits in L2: its loads take the evict-normal policy (the row copy reads it
                           // next), else evict-first
    uint32_t tmem_cols;
    uint32_t exch_off;     // byte offset of the epilogue exchange area (from the aligned base)
    uint32_t win_off;      // byte offset of the per-token winning logits
    uint32_t staging_off;  // split mode: byte offset of the DSMEM staging area
    uint32_t tail_off;     // byte offset of TcSmemTail
    int staging_alias;     // split mode: the staging area overlays the TMA ring
    // route + dispatch in one launch (split mode, every CTA resident): the counting
    // sort of the launch's slots and the bf16 row copy after a grid barrier
    int32_t *d_counts, *d_offsets, *d_row_map, *d_src_slot;
    const uint4 *d_X;      // X as 16-byte chunks
    uint4 *d_Xp;           // [N*K, H] bf16 rows in expert order, or nullptr
    unsigned *d_bar;       // [0] arrive, [1] depart: zero before the launch, returned to zero
    int32_t *d_hist;       // [CTAs][E] slot count per CTA and expert
    int d_prefetch;        // the CTA's X rows are bulk-copied to shared memory offset 0 first
    uint32_t d_scr_off;    // byte offset of the dispatch scratch (an mbarrier, then the counts)
};

// Row stride (floats) of the split-mode staging buffer: NP + 4 keeps rows
// 16-byte aligned for vector DSMEM stores and spreads banks.
__host__ __device__ constexpr int stage_row_floats(int NP) { return NP + 4; }

// Epilogue exchange area (persistent mode): per column part a sorted list per
// token (KMAX keys + KMAX ids) and the running (max, sum-exp); then, in both
// modes, per token the final K logits.
__host__ __device__ constexpr uint32_t exch_lists_bytes(int kmax, int nparts)
{
    return static_cast<uint32_t>(nparts * kBM * kmax * 8 + nparts * kBM * 2 * 4);
}
// Selection window: per token the K selected logits (then the weights) and the
// K selected ids, token-minor ([KMAX][128] floats, then [KMAX][128] ints), from
// which the outputs leave with coalesced stores.
__host__ __device__ constexpr uint32_t win_bytes(int kmax) { return static_cast<uint32_t>(2 * kBM * kmax * 4); }

// Coalesced copy of `rows` consecutive tokens' K values from a token-minor
// window (value k of token r at win[k * kBM + r0 + r]) to dst[r * K + k]; the
// `nthr` threads with rank `t` share the copy.
template <typename T>
__device__ __forceinline__ void window_to_global(T *dst, const T *win, int r0, int rows, int K, int t, int nthr)
{
    const int total = rows * K;
    int k = t % K, r = t / K;
    const int dk = nthr % K, dr = nthr / K;
    for (int i = t; i < total; i += nthr) {
        dst[i] = win[k * kBM + r0 + r];
        k += dk;
        r += dr;
        if (k >= K) {
            k -= K;
            ++r;
        }
    }
}

// Logits are ranked by an order-preserving int32 key (canon_key below: keys
// compare like the floats, with NaN taken as -inf and no -0 reaching it).
// kKeyEmpty (below the key of -inf) marks an empty list slot.
constexpr int kKeyEmpty = static_cast<int>(0x80000000u);

__device__ __forceinline__ float key_value(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7FFFFFFF)); }

// (ka, ia) ranks above (kb, ib): larger logit, or equal logit and lower expert id.
__device__ __forceinline__ bool ranks_above(int ka, int ia, int kb, int ib)
{
    return ka > kb || (ka == kb && ia < ib);
}

// Insert a candidate into a sorted top-KMAX list (keys descending).  The
// candidate's id is larger than every id already in the list (candidates
// arrive in increasing id order), so it goes below all equal keys: slot t
// takes the candidate where it is the first slot with key < new key, the entry
// above it where a slot above was already displaced, else keeps its own.
// Every slot decides from the old list alone: no branches, no carried chain.
template <int KMAX>
__device__ __forceinline__ void topk_push(int (&k)[KMAX], int (&ix)[KMAX], int nk, int ne)
{
    bool prev = false;
    int pk = kKeyEmpty, pi = kEmpty;
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
        const bool c = nk > k[t];
        const int ok = k[t], oi = ix[t];
        k[t] = c ? (prev ? pk : nk) : ok;
        ix[t] = c ? (prev ? pi : ne) : oi;
        prev = c;
        pk = ok;
        pi = oi;
    }
}

template <int KMAX>
__device__ __forceinline__ void topk_clear(int (&k)[KMAX], int (&ix)[KMAX])
{
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
        k[t] = kKeyEmpty;
        ix[t] = kEmpty;
    }
}

// Drop the head of a sorted list (shift up by one).
template <int KMAX>
__device__ __forceinline__ void topk_pop_if(int (&k)[KMAX], int (&ix)[KMAX], bool pop)
{
#pragma unroll
    for (int t = 0; t + 1 < KMAX; ++t) {
        k[t] = pop ? k[t + 1] : k[t];
        ix[t] = pop ? ix[t + 1] : ix[t];
    }
    k[KMAX - 1] = pop ? kKeyEmpty : k[KMAX - 1];
    ix[KMAX - 1] = pop ? kEmpty : ix[KMAX - 1];
}

__device__ __forceinline__ float logit_of(float acc, float bias)
{
    const float x = acc + bias;
    return isnan(x) ? -INFINITY : x;
}

// The logit acc + bias with NaN as -inf, and its order key, for a bias that is
// never -0 (the kernel stores bias + 0.0f): then the sum is never -0 either (in
// round-to-nearest a sum is -0 only when both terms are), so the key needs no
// sign-of-zero fix, and fmaxf(NaN, -inf) = -inf takes care of NaN.
__device__ __forceinline__ float canon_logit(float acc, float bias_canon)
{
    return fmaxf(acc + bias_canon, -INFINITY);
}

__device__ __forceinline__ int canon_key(float x)
{
    const int b = __float_as_int(x);
    return b ^ ((b >> 31) & 0x7FFFFFFF);
}

// Merge two sorted top-K lists held in shared memory (keys and ids at a stride
// of kBM ints) into the first K entries of registers: K rounds of "take the
// better head", equal keys to the lower id.
template <int KMAX>
__device__ __forceinline__ void merge2_to_regs(const int *ka_s, const int *ia_s, const int *kb_s, const int *ib_s, int K,
                                               int (&k)[KMAX], int (&ix)[KMAX])
{
    int pa = 0, pb = 0;
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
        if (t < K) {
            const int ka = pa < K ? ka_s[pa * kBM] : kKeyEmpty;
            const int ia = pa < K ? ia_s[pa * kBM] : kEmpty;
            const int kb = pb < K ? kb_s[pb * kBM] : kKeyEmpty;
            const int ib = pb < K ? ib_s[pb * kBM] : kEmpty;
            const bool take_b = ranks_above(kb, ib, ka, ia);
            k[t] = take_b ? kb : ka;
            ix[t] = take_b ? ib : ia;
            pa += take_b ? 0 : 1;
            pb += take_b ? 1 : 0;
        }
    }
}

// Online max / sum of exp over the logits a thread sees (renorm off, or the
// logsumexp requested).  The terms use the hardware exponential (__expf, a few
// ulp): the full softmax denominator feeds only the renorm-off weights and the
// logsumexp, where a relative error of ~1e-7 is far below their tolerance.
__device__ __forceinline__ void online_sumexp(float x, float &r, float &z)
{
    if (x == -INFINITY) return;
    if (x > r) {
        z = z * __expf(r - x) + 1.f;
        r = x;
    } else {
        z += __expf(x - r);
    }
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_addr, uint32_t cta)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(cta));
    return r;
}

__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, float a, float b, float c, float d)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Dispatch of a split-mode launch's own tokens, run by all threads of every CTA
// once its top-K ids are in global memory: CTA c = tile * S + rank owns tokens
// [c R, c R + R) (R = kBM / S), so the CTAs in index order hold the slots in
// token order.  Per-warp ballot histograms give each slot its rank among the
// CTA's slots of the same expert (stable in slot order); the CTA's counts go to
// the grid-wide table, a bounded grid barrier follows, then every CTA sums the
// table (all CTAs: expert totals; lower CTAs: rows before its own), forms the
// exclusive prefix, writes row_map (and src_slot), and copies its tokens' rows
// into X_perm.  All of `smem` is free by then: with p.d_prefetch the CTA's rows
// (contiguous in X) are bulk-copied to offset 0 before the barrier and leave as
// one bulk store per destination row; the counts and an mbarrier live at
// p.d_scr_off.
template <int KMAX>
__device__ __forceinline__ void fused_dispatch_tail(const TcParams &p, unsigned char *smem)
{
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int E = p.E;
    const int K = p.K;
    const int S = p.nsplit;
    const int R = kBM / S;
    const int c = static_cast<int>(blockIdx.y) * S + static_cast<int>(blockIdx.x);
    const unsigned G = gridDim.x * gridDim.y;
    const int64_t n0 = static_cast<int64_t>(c) * R;
    const int64_t left = p.N - n0;
    const int ntok = left <= 0 ? 0 : (left < R ? static_cast<int>(left) : R);
    const int ns = ntok * K;
    const int64_t s0 = n0 * K;
    uint64_t *pf_bar = reinterpret_cast<uint64_t *>(smem + p.d_scr_off);
    int *wcnt = reinterpret_cast<int *>(smem + p.d_scr_off + 16);   // [kWarps][E]
    int *total = wcnt + kWarps * E;    // [E]
    int *before = total + E;           // [E]
    int *offset = before + E;          // [E + 1]
    int *rows_s = offset + E + 1;      // [ns]
    int *flag = rows_s + R * K;        // [1]
    const int per_warp = (ns + kWarps - 1) / kWarps;
    const int w0 = min(ns, per_warp * warp);
    const int w1 = min(ns, w0 + per_warp);
    int *my_cnt = wcnt + warp * E;

    const int chunks = p.H >> 3;
    const bool pf = p.d_prefetch && p.d_Xp != nullptr && ntok > 0;
    // this warp's slot ids (slot i = token i / K, rank i % K), as the epilogue
    // left them in the selection window, in registers before the row prefetch
    // may overwrite that memory; ids outside [0, E) become E (skipped)
    constexpr int kIdIters = ((kBM / 2 * KMAX + kWarps - 1) / kWarps + 31) / 32;   // R <= kBM / 2
    int ids[kIdIters];
    {
        const int *ids_s = reinterpret_cast<const int *>(smem + p.win_off) + KMAX * kBM;   // the id window
#pragma unroll
        for (int j = 0; j < kIdIters; ++j) {
            const int i = w0 + lane + 32 * j;
            int e = E;
            if (i < w1) {
                const int t = i / K;
                e = ids_s[(i - t * K) * kBM + t];
            }
            ids[j] = (e < 0 || e >= E) ? E : e;
        }
    }
    // the rows this CTA will copy do not depend on the dispatch: start their
    // bulk copy into shared memory now (the router is done with all of it)
    fence_proxy_async_smem();
    __syncthreads();
    if (pf && tid == 0) {
        mbar_init(pf_bar, 1);
        fence_mbarrier_init();
        mbar_arrive_expect_tx(pf_bar, static_cast<uint32_t>(ntok) * chunks * 16u);
        bulk_load(smem, p.d_X + n0 * chunks, static_cast<uint32_t>(ntok) * chunks * 16u, pf_bar);  // rows are contiguous
    }
    for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
    for (int e = tid; e < E; e += kThreads) {
        total[e] = 0;
        before[e] = 0;
    }
    __syncthreads();
    // per-warp histograms of contiguous slot ranges
#pragma unroll
    for (int j = 0; j < kIdIters; ++j) {
        if (w0 + 32 * j < w1) {   // warp-uniform
            const int e = ids[j];
            const uint32_t peers = same_key_lanes(e);
            if (e < E && lane == __ffs(peers) - 1) my_cnt[e] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        int run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int v = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += v;
        }
        p.d_hist[static_cast<int64_t>(c) * E + e] = run;
    }

    // grid barrier (bounded): every CTA arrives, whatever happened before
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        red_add_release_gpu(&p.d_bar[0], 1u);
        const uint64_t tb = globaltimer_ns();
        int ok = 1;
        for (uint32_t it = 0; ld_acquire_gpu(&p.d_bar[0]) < G; ++it) {
            if ((it & 255u) == 255u && globaltimer_ns() - tb > kWaitLimitNs) {
                ok = 0;
                break;
            }
        }
        *flag = ok;
    }
    __syncthreads();
    if (!*flag) {
        if (tid == 0) report_status(p.status, MOE_ERR_TIMEOUT);
        if (pf) {   // let the row copy land before the CTA exits
            volatile int no_abort = 0;
            mbar_wait_bounded(pf_bar, 0, &no_abort);
        }
        return;
    }

    // expert totals and the rows of lower CTAs: thread (grp, four experts q) sums
    // table rows grp, grp + groups, ... as 16-byte vectors (E % 8 == 0 on this
    // path; rows are E ints apart), eight loads in flight before the first add
    {
        const int nq = E >> 2;
        const int groups = kThreads / nq;   // >= 5 (E <= 256)
        const int q = tid % nq;
        const int grp = tid / nq;
        if (grp < groups) {
            const int4 *tab = reinterpret_cast<const int4 *>(p.d_hist);
            int tot[4] = {0, 0, 0, 0}, bef[4] = {0, 0, 0, 0};
            for (int c0 = grp; c0 < static_cast<int>(G); c0 += 8 * groups) {
                int4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int cc = c0 + u * groups;
                    v[u] = cc < static_cast<int>(G) ? __ldcg(tab + static_cast<int64_t>(cc) * nq + q)
                                                     : make_int4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const bool lower = c0 + u * groups < c;
                    const int w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        tot[t] += w4[t];
                        bef[t] += lower ? w4[t] : 0;
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                atomicAdd(&total[4 * q + t], tot[t]);
                atomicAdd(&before[4 * q + t], bef[t]);
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive prefix over the experts, eight per lane
        int vals[8];
        int local = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            vals[i] = e < E ? total[e] : 0;
            local += vals[i];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - local;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            if (e < E) offset[e] = run;
            run += vals[i];
        }
        if (lane == 31) offset[E] = incl;
    }
    __syncthreads();
    if (c == 0) {
        for (int e = tid; e <= E; e += kThreads) {
            p.d_offsets[e] = offset[e];
            if (e < E) p.d_counts[e] = total[e];
        }
    }
    for (int i = tid; i < kWarps * E; i += kThreads) {
        const int e = i % E;
        wcnt[i] += offset[e] + before[e];
    }
    __syncthreads();

    // stable scatter: slot i of this CTA gets row offset + before + its rank
#pragma unroll
    for (int j = 0; j < kIdIters; ++j) {
        if (w0 + 32 * j < w1) {   // warp-uniform
            const int i = w0 + 32 * j + lane;
            const int e = ids[j];
            const uint32_t peers = same_key_lanes(e);
            const uint32_t below = peers & ((1u << lane) - 1u);
            if (i < w1) {
                const int r = e < E ? my_cnt[e] + __popc(below) : -1;
                rows_s[i] = r;
                p.d_row_map[s0 + i] = r;
                if (e < E && p.d_src_slot) p.d_src_slot[r] = static_cast<int32_t>(s0 + i);
            }
            __syncwarp();
            if (e < E && below == 0) my_cnt[e] += __popc(peers);
            __syncwarp();
        }
    }

    // the last CTA to leave returns the barrier counters to zero
    if (tid == 0) {
        const unsigned old = atomicAdd(&p.d_bar[1], 1u);
        if (old == G - 1) {
            p.d_bar[0] = 0;
            p.d_bar[1] = 0;
            __threadfence();
        }
    }

    // rows of this CTA's tokens: where they were prefetched, one bulk store per
    // destination row (the TMA engine copies them out of shared memory); else one
    // warp per token from global memory (L2, where the router just streamed them)
    if (p.d_Xp != nullptr) {
        __syncthreads();
        if (pf) {
            // the copy depends on nothing but memory: wait for it (time-bounded)
            // whatever else went wrong, so that no copy is in flight at exit
            volatile int no_abort = 0;
            if (!mbar_wait_bounded(pf_bar, 0, &no_abort)) {
                if (tid == 0) report_status(p.status, MOE_ERR_TIMEOUT);
                return;
            }
            bool issued = false;
            for (int i = tid; i < ns; i += kThreads) {
                const int r = rows_s[i];
                if (r >= 0) {
                    bulk_store(p.d_Xp + static_cast<int64_t>(r) * chunks, smem + static_cast<size_t>(i / K) * chunks * 16,
                               static_cast<uint32_t>(chunks) * 16u);
                    issued = true;
                }
            }
            if (issued) bulk_commit_and_wait_all();
        } else {
            // eight 16-byte chunks per lane loaded before any of them is stored (the
            // stores may alias X as far as the compiler knows, so a plain loop would
            // keep one load in flight)
            constexpr int kCpl = 8;
            for (int j = warp; j < ntok; j += kWarps) {
                const uint4 *src = p.d_X + (n0 + j) * chunks;
                int rk[KMAX];
#pragma unroll
                for (int k = 0; k < KMAX; ++k) rk[k] = k < K ? rows_s[j * K + k] : -1;
                for (int base = 0; base < chunks; base += 32 * kCpl) {
                    uint4 v[kCpl];
#pragma unroll
                    for (int u = 0; u < kCpl; ++u) {
                        const int ch = base + lane + 32 * u;
                        v[u] = ch < chunks ? __ldg(src + ch) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int u = 0; u < kCpl; ++u) {
                        const int ch = base + lane + 32 * u;
                        if (ch < chunks) {
#pragma unroll
                            for (int k = 0; k < KMAX; ++k)
                                if (rk[k] >= 0) p.d_Xp[static_cast<int64_t>(rk[k]) * chunks + ch] = v[u];
                        }
                    }
                }
            }
        }
    }
    // (no dependents trigger: the next kernel is launched once every CTA has left,
    // so that its CTAs never share an SM with one of these, whose large
    // shared-memory carve-out they would inherit)
}

template <int KMAX, bool SPLIT, bool FUSE = false>
__global__ void __launch_bounds__(TcShape<KMAX, SPLIT>::kThr, SPLIT ? 2 : 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const TcParams p)
{
    static_assert(SPLIT || !FUSE, "the dispatch tail takes its ids from the split-mode epilogue");
    constexpr int EPW = TcShape<KMAX, SPLIT>::kEpi;    // epilogue warps
    constexpr int NT = TcShape<KMAX, SPLIT>::kThr;     // threads of the CTA
    constexpr int NPART = TcShape<KMAX, SPLIT>::kParts;
    static_assert(!FUSE || NT == kThreads, "the dispatch tail is written for the split-mode CTA");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms, as an offset from the
    // shared array: a pointer derived this way keeps its shared address space,
    // so the compiler emits shared-memory loads and stores rather than generic ones
    const uint32_t smem_pad = (1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u;
    unsigned char *smem = smem_raw + smem_pad;
    const uint32_t b_slot_bytes = static_cast<uint32_t>(p.EP) * kBK * 2;
    unsigned char *a_base = smem;
    unsigned char *b_base = smem + static_cast<size_t>(p.stages) * kABytes * (SPLIT ? 1 : p.kpack);
    TcSmemTail &tail = *reinterpret_cast<TcSmemTail *>(smem + p.tail_off);
    float *bias_s = reinterpret_cast<float *>(&tail + 1);
    int *hist_s = reinterpret_cast<int *>(bias_s + p.EP);                // [EP] selections per expert
    // exchange area, token-minor so that the lanes of a warp touch consecutive words
    int *lst_k = reinterpret_cast<int *>(smem + p.exch_off);            // [NPART][KMAX][128] keys
    int *lst_i = lst_k + NPART * kBM * KMAX;                               // [NPART][KMAX][128] ids
    float *lst_rz = reinterpret_cast<float *>(lst_i + NPART * kBM * KMAX); // [NPART][2][128]
    float *win_v = reinterpret_cast<float *>(smem + p.win_off);            // [KMAX][128] logits, then weights
    int *win_i = reinterpret_cast<int *>(win_v + KMAX * kBM);              // [KMAX][128] ids

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The split-K exchange writes into the shared memory of the other CTAs of the
    // cluster, so it runs only in clusters of the planned nsplit CTAs.  A launch
    // whose clusters were dropped (a profiler may run a cooperative cluster launch
    // with clusters of one CTA) runs "solo" instead: each CTA takes the whole H
    // range of its tile and finishes its own kBM / nsplit tokens, with no peer
    // memory touched.  The cluster size is the same for every CTA, so all of them
    // take the same branch before any barrier.
    bool solo = false;
    if constexpr (SPLIT) {
        uint32_t ncta;
        asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncta));
        solo = ncta != static_cast<uint32_t>(p.nsplit);
    }
    const uint32_t rank = SPLIT ? (solo ? blockIdx.x : cluster_rank()) : 0u;
    const int nk = (p.H + kBK - 1) / kBK;
    const int kb0 = SPLIT && !solo ? static_cast<int>(rank) * p.kb_per : 0;
    const int kb1 = SPLIT && !solo ? min(nk, kb0 + p.kb_per) : nk;
    const int nkb = kb1 > kb0 ? kb1 - kb0 : 0;    // K-steps of this CTA per tile (0: contributes nothing)
    const int first_tile = SPLIT ? static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.x);
    const int tile_step = SPLIT ? p.tiles : static_cast<int>(gridDim.x);  // split: exactly one tile
    const int K = p.K;
    const int E = p.E;
    volatile int *abort_flag = &tail.abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&tail.full[s], 1);
            mbar_init(&tail.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tail.acc_full[b], 1);
            mbar_init(&tail.acc_empty[b], EPW);
        }
        mbar_init(&tail.drain, 1);
        tail.abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(&tail.tmem_base, p.tmem_cols);
        tmem_relinquish();
    }
    // No early launch trigger (griddepcontrol.launch_dependents): the next
    // kernel in the stream is released when this grid completes.  An early
    // trigger gained nothing in a stream, and in a CUDA graph it staged the next
    // launch while these CTAs held every SM: the router itself then ran ~2 us
    // longer at 16384 x 2048 x 128 experts, and the next kernels' CTAs ran with
    // this kernel's large shared-memory carve-out, i.e. a small L1 for their
    // loads in flight (graph replay of the 65536 x 4096 step: 644 against 586 us
    // without the trigger).  With the dispatch fused in, the combine that follows
    // was likewise slower with a trigger at the end of the launch (4096 tokens:
    // 54.2 against 50.3 us per step).
    tc_fence_before_sync();
    __syncthreads();  // barriers initialised, TMEM allocated
    tc_fence_after_sync();
    // split mode with a staging area of its own: announce that this CTA runs
    // (peers wait for it before writing into its shared memory); the matching
    // wait comes after the MMAs
    if constexpr (SPLIT)
        if (!p.staging_alias) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const uint32_t tmem_base = tail.tmem_base;
    // inputs may come from the previous kernel in the stream (programmatic launch)
    pdl_wait_prior_grids();
    if (warp != 0) {
        // the producer starts streaming at once; the bias is needed by the epilogue only
        for (int e = threadIdx.x - 32; e < p.EP; e += NT - 32) {
            // + 0.0f turns a -0 bias into +0 (see canon_logit)
            bias_s[e] = ((p.bias != nullptr && e < E) ? p.bias[e] : 0.f) + 0.0f;
            hist_s[e] = 0;
        }
        named_barrier_sync(7, NT - 32);
    }

    bool acc_ok = false;  // split mode, epilogue threads: the partial accumulator is complete
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // (the ring slot and its phase advance by counters: this thread paces the
        // stream, so its loop is kept free of divisions)
        if (lane == 0) {
            const uint64_t pol_x = p.x_keep ? l2_policy_evict_normal() : l2_policy_evict_first();
            const uint64_t pol_w = l2_policy_evict_last();
            const int kp = SPLIT ? 1 : p.kpack;   // K-steps per ring stage
            const int nst = (nkb + kp - 1) / kp;   // ring stages per tile
            const uint32_t stage_a = kABytes * kp, stage_b = b_slot_bytes * kp;
            const int nwb = p.EP / 64;             // gate-weight boxes per stage
            uint32_t g = 0, s = 0, ph = 0;         // stages issued (across tiles), ring slot, its phase
            bool stop = false;
            for (int tile = first_tile; tile < p.tiles && !stop; tile += tile_step) {
                const int m0 = tile * p.tile_rows;
                for (int i = 0; i < nst; ++i) {
                    if (!mbar_wait_bounded(&tail.empty[s], ph ^ 1u, abort_flag)) {
                        stop = true;
                        break;
                    }
                    uint64_t *fb = &tail.full[s];
                    unsigned char *as = a_base + s * stage_a;
                    unsigned char *bs = b_base + s * stage_b;
                    mbar_arrive_expect_tx(fb, stage_a + stage_b);
                    if (kp == 1) {
                        const int kc = (kb0 + i) * kBK;
                        tma_load_2d(as, &tmX, fb, kc, m0, pol_x);
                        for (int jw = 0; jw < nwb; ++jw) tma_load_2d(bs + jw * kBBoxBytes, &tmW, fb, jw * 64, kc, pol_w);
                    } else {
                        // two K-steps: one 3D box of X ([2 column blocks][kBM rows][64]) and one
                        // [128 K-rows x 64 experts] box of the gate weight per 64 experts
                        tma_load_3d(as, &tmX, fb, 0, m0, 2 * i, pol_x);
                        for (int jw = 0; jw < nwb; ++jw)
                            tma_load_2d(bs + jw * 2 * kBBoxBytes, &tmW, fb, jw * 64, 2 * i * kBK, pol_w);
                    }
                    ++g;
                    if (++s == static_cast<uint32_t>(p.stages)) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // let the copies already issued land before the shared memory is reused
                const uint32_t from = g > static_cast<uint32_t>(p.stages) ? g - p.stages : 0u;
                for (uint32_t x = from; x < g; ++x) {
                    volatile int no_abort = 0;
                    mbar_wait_bounded(&tail.full[x % p.stages], (x / p.stages) & 1u, &no_abort);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // (as the producer: counters for the ring, and descriptors of slot 0 to which a
        // slot's byte offset >> 4 is added in the start-address field)
        if (lane == 0) {
            const uint32_t idesc = make_idesc_bf16_f32(kBM, static_cast<uint32_t>(p.NP), 0u, 1u);
            const int kp = SPLIT ? 1 : p.kpack;
            const int nst = (nkb + kp - 1) / kp;
            const uint32_t stage_a = kABytes * kp, stage_b = b_slot_bytes * kp;
            // A: K-major, 128-byte rows, 8-row groups 1024 B apart; +32 B per K=16 step, the
            // next 64-column block kABytes further on.  B: MN-major, 64-expert atoms kp x 8 KiB
            // apart (LBO), 8-row K groups 1024 B apart (SBO); +16 rows x 128 B per K=16 step.
            const uint64_t a_desc0 = make_smem_desc_sw128(smem_u32(a_base), 16, 1024);
            const uint64_t b_desc0 = make_smem_desc_sw128(smem_u32(b_base), kp * kBBoxBytes, 1024);
            uint32_t s = 0, ph = 0;
            int j = 0;
            bool stop = false;
            for (int tile = first_tile; tile < p.tiles; tile += tile_step, ++j) {
                const int b = j & 1;
                if (!mbar_wait_bounded(&tail.acc_empty[b], ((j >> 1) & 1) ^ 1, abort_flag)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * p.NP);
                for (int i = 0; i < nst; ++i) {
                    if (!mbar_wait_bounded(&tail.full[s], ph, abort_flag)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t ad = a_desc0 + ((s * stage_a) >> 4);
                    const uint64_t bd = b_desc0 + ((s * stage_b) >> 4);
                    const uint32_t acc0 = i != 0 ? 1u : 0u;
                    if (kp == 1) {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            tc_mma_f16(d_tmem, ad + kk * 2, bd + kk * 128, idesc, kk != 0 ? 1u : acc0);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 2 * (kBK / 16); ++kk)
                            tc_mma_f16(d_tmem, ad + (kk >> 2) * (kABytes >> 4) + (kk & 3) * 2, bd + kk * 128, idesc,
                                       kk != 0 ? 1u : acc0);
                    }
                    tc_commit(&tail.empty[s]);  // slot free once these MMAs have read it
                    if (++s == static_cast<uint32_t>(p.stages)) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (stop) break;
                tc_commit(&tail.acc_full[b]);   // this tile's logits (or partial logits) complete
            }
            tc_commit(&tail.drain);
            volatile int no_abort = 0;
            mbar_wait_bounded(&tail.drain, 0, &no_abort);
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q = warp & 3;                // TMEM lane quarter this warp may access
        const int h = (warp - 2) >> 2;         // which part of the expert columns
        const int row = q * 32 + lane;         // token row of the tile (= TMEM lane)
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        if constexpr (!SPLIT) {
            const int npp = p.NP / NPART;      // columns per part (a multiple of 4)
            int j = 0;
            for (int tile = first_tile; tile < p.tiles; tile += tile_step, ++j) {
                const int b = j & 1;
                // (a vote, so that the warp leaves the wait together: lanes that left the
                // polling loop at different times would otherwise run what follows apart)
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tail.acc_full[b], (j >> 1) & 1, abort_flag, 64)))
                    break;
                tc_fence_after_sync();
                // ---- this part's columns: two interleaved lists for ILP
                int ak[KMAX], bk[KMAX], ai[KMAX], bi[KMAX];
                topk_clear<KMAX>(ak, ai);
                topk_clear<KMAX>(bk, bi);
                float r = -INFINITY, z = 0.f;
                const int c_end = min(E, h * npp + npp);
                const uint32_t col_addr = lane_addr + static_cast<uint32_t>(b * p.NP);
                int c = h * npp;
                // 32 columns per TMEM round trip while they lie inside this part, then 8, then 4
#pragma unroll 1
                for (; c + 32 <= c_end; c += 32) {
                    float v[32];
                    tmem_ld_32x32b_x32(col_addr + c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 32; t += 2) {
                        const float x0 = canon_logit(v[t], bias_s[c + t]);
                        const float x1 = canon_logit(v[t + 1], bias_s[c + t + 1]);
                        topk_push<KMAX>(ak, ai, canon_key(x0), c + t);
                        topk_push<KMAX>(bk, bi, canon_key(x1), c + t + 1);
                        if (p.need_z) {
                            online_sumexp(x0, r, z);
                            online_sumexp(x1, r, z);
                        }
                    }
                }
#pragma unroll 1
                for (; c + 8 <= c_end; c += 8) {
                    float v[8];
                    tmem_ld_32x32b_x8(col_addr + c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 8; t += 2) {
                        const float x0 = canon_logit(v[t], bias_s[c + t]);
                        const float x1 = canon_logit(v[t + 1], bias_s[c + t + 1]);
                        topk_push<KMAX>(ak, ai, canon_key(x0), c + t);
                        topk_push<KMAX>(bk, bi, canon_key(x1), c + t + 1);
                        if (p.need_z) {
                            online_sumexp(x0, r, z);
                            online_sumexp(x1, r, z);
                        }
                    }
                }
                if (c < c_end) {   // a last group of 4 columns (E % 8 == 0, parts start at multiples of 4)
                    float v[4];
                    tmem_ld_32x32b_x4(col_addr + c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 4; t += 2) {
                        const float x0 = canon_logit(v[t], bias_s[c + t]);
                        const float x1 = canon_logit(v[t + 1], bias_s[c + t + 1]);
                        topk_push<KMAX>(ak, ai, canon_key(x0), c + t);
                        topk_push<KMAX>(bk, bi, canon_key(x1), c + t + 1);
                        if (p.need_z) {
                            online_sumexp(x0, r, z);
                            online_sumexp(x1, r, z);
                        }
                    }
                }
                // the accumulator may be overwritten by the next tile's MMAs from here on
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tail.acc_empty[b]);
                // ---- merge the two lists into this part's sorted top-K (shared memory)
                int *my_k = lst_k + h * KMAX * kBM + row;
                int *my_i = lst_i + h * KMAX * kBM + row;
#pragma unroll 1
                for (int k = 0; k < K; ++k) {
                    const bool take_b = ranks_above(bk[0], bi[0], ak[0], ai[0]);
                    my_k[k * kBM] = take_b ? bk[0] : ak[0];
                    my_i[k * kBM] = take_b ? bi[0] : ai[0];
                    topk_pop_if<KMAX>(ak, ai, !take_b);
                    topk_pop_if<KMAX>(bk, bi, take_b);
                }
                lst_rz[(h * 2) * kBM + row] = r;
                lst_rz[(h * 2 + 1) * kBM + row] = z;
                named_barrier_sync(1 + q, 32 * NPART);   // every part's list is ready
                if constexpr (NPART == 4) {
                    // parts 0 and 2 fold in parts 1 and 3 (written back over their own lists)
                    if ((h & 1) == 0) {
                        merge2_to_regs<KMAX>(my_k, my_i, my_k + KMAX * kBM, my_i + KMAX * kBM, K, ak, ai);
#pragma unroll
                        for (int t = 0; t < KMAX; ++t)
                            if (t < K) {
                                my_k[t * kBM] = ak[t];
                                my_i[t * kBM] = ai[t];
                            }
                        if (p.need_z) {
                            const float r1 = lst_rz[(h * 2 + 2) * kBM + row], z1 = lst_rz[(h * 2 + 3) * kBM + row];
                            const float rm = fmaxf(r, r1);
                            const float zs = (z > 0.f ? z * expf(r - rm) : 0.f) + (z1 > 0.f ? z1 * expf(r1 - rm) : 0.f);
                            lst_rz[(h * 2) * kBM + row] = rm;
                            lst_rz[(h * 2 + 1) * kBM + row] = zs;
                        }
                    }
                    named_barrier_sync(1 + q, 32 * NPART);
                }
                if (h == 0) {
                    // ---- two-way merge of the halves, K rounds; ids written as selected
                    constexpr int kOther = NPART / 2;   // the part holding the other half's list
                    const int n = tile * p.tile_rows + row;
                    // rows past tile_rows belong to the next tile (the TMA box is kBM rows)
                    const bool mine = row < p.tile_rows && n < p.N;
                    const int *ok = lst_k + kOther * KMAX * kBM + row;
                    const int *oi = lst_i + kOther * KMAX * kBM + row;
                    float *wrow = win_v + row;
                    int *irow = win_i + row;
                    int pa = 0, pb = 0;
#pragma unroll 1
                    for (int k = 0; k < K; ++k) {
                        const int ka = pa < K ? my_k[pa * kBM] : kKeyEmpty;
                        const int ia = pa < K ? my_i[pa * kBM] : kEmpty;
                        const int kb = pb < K ? ok[pb * kBM] : kKeyEmpty;
                        const int ib = pb < K ? oi[pb * kBM] : kEmpty;
                        const bool take_b = ranks_above(kb, ib, ka, ia);
                        wrow[k * kBM] = key_value(take_b ? kb : ka);
                        const int sel = take_b ? ib : ia;
                        irow[k * kBM] = sel;
                        if (mine && p.counts && sel < E) atomicAdd(hist_s + sel, 1);
                        pa += take_b ? 0 : 1;
                        pb += take_b ? 1 : 0;
                    }
                    const float m = wrow[0];   // the largest logit
                    float zfull = 0.f;         // sum over all experts of exp(logit - m)
                    if (p.need_z) {
                        const float r0 = lst_rz[row], z0 = lst_rz[kBM + row];
                        const float r1 = lst_rz[(kOther * 2) * kBM + row], z1 = lst_rz[(kOther * 2 + 1) * kBM + row];
                        zfull = (z0 > 0.f ? z0 * expf(r0 - m) : 0.f) + (z1 > 0.f ? z1 * expf(r1 - m) : 0.f);
                    }
                    // the window's logits become exp(logit - m), then the weights
                    float denom = zfull;
                    if (p.renorm) denom = 0.f;
#pragma unroll 1
                    for (int k = 0; k < K; ++k) {
                        const float e = expf(wrow[k * kBM] - m);
                        wrow[k * kBM] = e;
                        if (p.renorm) denom += e;
                    }
#pragma unroll 1
                    for (int k = 0; k < K; ++k) wrow[k * kBM] = wrow[k * kBM] / denom;
                    if (mine && p.lse) p.lse[n] = m == -INFINITY ? -INFINITY : m + logf(zfull);
                    // this quarter's tokens leave with coalesced stores (the warp holds them all)
                    __syncwarp();
                    const int r0 = q * 32;
                    const int64_t n0 = static_cast<int64_t>(tile) * p.tile_rows + r0;
                    const int64_t left = min(static_cast<int64_t>(p.tile_rows - r0), p.N - n0);
                    const int vr = left <= 0 ? 0 : (left < 32 ? static_cast<int>(left) : 32);
                    window_to_global<int>(p.topk_idx + n0 * K, win_i, r0, vr, K, lane, 32);
                    window_to_global<float>(p.topk_w + n0 * K, win_v, r0, vr, K, lane, 32);
                }
                named_barrier_sync(1 + q, 32 * NPART);   // the lists have been consumed
            }
        } else {
            acc_ok = __all_sync(0xffffffffu, mbar_wait_bounded(&tail.acc_full[0], 0, abort_flag, 64));
            tc_fence_after_sync();
        }
    }

    if constexpr (SPLIT) {
        // ------------------------------------------------------------ split-K reduction through DSMEM
        const int S = p.nsplit;
        const int R = kBM / S;                          // tokens owned by each CTA of the cluster
        const int RS = stage_row_floats(p.NP);
        float *buf = reinterpret_cast<float *>(smem + p.staging_off);  // [S slices][R rows][RS]
        __syncwarp();
        if (p.staging_alias)
            cluster_sync_all();  // every CTA's MMAs are complete, so its ring may be overwritten
        else  // every CTA of the cluster has started, so its staging area may be written
            asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        if (warp >= 2 && acc_ok && nkb > 0) {
            const int q = warp & 3;
            const int h = (warp - 2) >> 2;
            const int row = q * 32 + lane;
            const int nph = p.NP >> 1;
            const uint32_t owner = static_cast<uint32_t>(row / R);
            // solo: the CTA's own rows go to slice 0 of its own staging area (the
            // shared::cta address of an own-CTA location is valid for st.shared::cluster)
            const uint32_t local = smem_u32(buf + ((solo ? 0 : static_cast<int>(rank)) * R + row % R) * RS);
            const uint32_t remote = solo ? local : dsmem_map(local, owner);
            const bool send = !solo || owner == rank;   // (the TMEM loads stay warp-wide)
            const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            int c = h * nph;
#pragma unroll 1
            for (; c + 32 <= h * nph + nph; c += 32) {
                float v[32];
                tmem_ld_32x32b_x32(lane_addr + c, v);
                tmem_ld_wait();
                if (send) {
#pragma unroll
                    for (int g = 0; g < 32; g += 4)
                        st_dsmem_v4(remote + (c + g) * 4, v[g], v[g + 1], v[g + 2], v[g + 3]);
                }
            }
#pragma unroll 1
            for (; c < h * nph + nph; c += 8) {
                float v[8];
                tmem_ld_32x32b_x8(lane_addr + c, v);
                tmem_ld_wait();
                if (send) {
                    st_dsmem_v4(remote + c * 4, v[0], v[1], v[2], v[3]);
                    st_dsmem_v4(remote + c * 4 + 16, v[4], v[5], v[6], v[7]);
                }
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        cluster_sync_all();                             // #2: all partial logits delivered
        if (warp >= 2) {
            const int t = threadIdx.x - 64;             // 0..255
            const int G = (32 * EPW) / R;               // threads per token: 2S (4, 8 or 16)
            const int lrow = t / G;
            const int part = t % G;
            const int n = first_tile * p.tile_rows + static_cast<int>(rank) * R + lrow;
            // CTAs that had K-steps (solo: this CTA alone, over all of H)
            const int nslices = solo ? 1 : min(S, (nk + p.kb_per - 1) / p.kb_per);
            const float *rowbuf = buf + lrow * RS;
            const int sstride = R * RS;                 // floats between the slices of a row
            // this thread's columns part, part + G, ...: eight per step with the loads
            // issued first, alternately into two lists (each sees increasing ids)
            int ak[KMAX], ai[KMAX], bk[KMAX], bi[KMAX];
            topk_clear<KMAX>(ak, ai);
            topk_clear<KMAX>(bk, bi);
            int col = part;
#pragma unroll 1
            for (; col + 7 * G < E; col += 8 * G) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c)   // summed in slice order
                    if (c < nslices) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) x[u] += rowbuf[c * sstride + col + u * G];
                    }
#pragma unroll
                for (int u = 0; u < 8; u += 2) {
                    topk_push<KMAX>(ak, ai, canon_key(canon_logit(x[u], bias_s[col + u * G])), col + u * G);
                    // (K > 8: one list, to stay within the registers of two CTAs per SM)
                    if constexpr (KMAX <= 8)
                        topk_push<KMAX>(bk, bi, canon_key(canon_logit(x[u + 1], bias_s[col + (u + 1) * G])),
                                        col + (u + 1) * G);
                    else
                        topk_push<KMAX>(ak, ai, canon_key(canon_logit(x[u + 1], bias_s[col + (u + 1) * G])),
                                        col + (u + 1) * G);
                }
            }
#pragma unroll 1
            for (; col < E; col += G) {
                float x = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (c < nslices) x += rowbuf[c * sstride + col];
                topk_push<KMAX>(ak, ai, canon_key(canon_logit(x, bias_s[col])), col);
            }
            // K rounds of selection across the 2G lists of the token (warp shuffles
            // between its G threads); the winner's list drops its head
            float *wrow = win_v + lrow;
            float m = 0.f;
#pragma unroll 1
            for (int k = 0; k < K; ++k) {
                const bool from_b = ranks_above(bk[0], bi[0], ak[0], ai[0]);
                int v = from_b ? bk[0] : ak[0];
                int i = from_b ? bi[0] : ai[0];
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) {
                    if (o < G) {
                        const int ov = __shfl_xor_sync(0xffffffffu, v, o);
                        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
                        const bool up = ranks_above(ov, oi, v, i);
                        v = up ? ov : v;
                        i = up ? oi : i;
                    }
                }
                const float fv = key_value(v);
                if (k == 0) m = fv;
                topk_pop_if<KMAX>(ak, ai, ai[0] == i);
                topk_pop_if<KMAX>(bk, bi, bi[0] == i);
                if (part == 0) {
                    wrow[k * kBM] = fv;
                    win_i[k * kBM + lrow] = i;   // also read by the dispatch tail
                    if (n < p.N && p.counts && i < E) atomicAdd(hist_s + i, 1);
                }
            }
            float z = 0.f;
            if (p.need_z) {
#pragma unroll 1
                for (int col = part; col < E; col += G) {
                    float x = 0.f;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        if (c < nslices) x += rowbuf[c * R * RS + col];
                    x = logit_of(x, bias_s[col]);
                    if (x != -INFINITY) z += __expf(x - m);
                }
#pragma unroll 1
                for (int o = G >> 1; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            }
            if (part == 0) {
                // the window's logits become exp(logit - m), then the weights
                float denom = p.renorm ? 0.f : z;
#pragma unroll 1
                for (int k = 0; k < K; ++k) {
                    const float e = expf(wrow[k * kBM] - m);
                    wrow[k * kBM] = e;
                    if (p.renorm) denom += e;
                }
#pragma unroll 1
                for (int k = 0; k < K; ++k) wrow[k * kBM] = wrow[k * kBM] / denom;
                if (n < p.N && p.lse) p.lse[n] = m == -INFINITY ? -INFINITY : m + logf(z);
            }
            // the CTA's R consecutive tokens leave with coalesced stores
            named_barrier_sync(6, 32 * kEpiWarps);
            const int64_t n0 = static_cast<int64_t>(first_tile) * p.tile_rows + static_cast<int64_t>(rank) * R;
            const int64_t left = p.N - n0;
            const int vr = left <= 0 ? 0 : (left < R ? static_cast<int>(left) : R);
            window_to_global<int>(p.topk_idx + n0 * K, win_i, 0, vr, K, t, 32 * kEpiWarps);
            window_to_global<float>(p.topk_w + n0 * K, win_v, 0, vr, K, t, 32 * kEpiWarps);
        }
    }

    __syncthreads();
    if (p.counts) {
        // this CTA's selections per expert, added to the grid-wide counts
        for (int e = threadIdx.x; e < E; e += NT)
            if (hist_s[e] != 0) atomicAdd(p.counts + e, hist_s[e]);
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
    if (threadIdx.x == 0 && tail.abort) report_status(p.status, MOE_ERR_TIMEOUT);
    if constexpr (FUSE) fused_dispatch_tail<KMAX>(p, smem);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

bool encode_2d_bf16(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                    uint32_t box_outer)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// X [N, H] viewed as [H/64 column blocks][N rows][64]: a box of 2 blocks x rows x
// 64 lands in shared memory as two [rows x 64] 128-byte-swizzled tiles back to
// back, i.e. two K-steps of the A operand in one copy.  Needs H % 64 == 0 (so
// that the blocks tile the rows exactly); false if the driver refuses the map.
bool encode_x_3d(CUtensorMap *map, const void *base, uint64_t H, uint64_t N, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn || H % 64 != 0) return false;
    const cuuint64_t dims[3] = {64, N, H / 64};
    const cuuint64_t strides[2] = {H * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int kmax_for(int K) { return K <= 2 ? 2 : K <= 4 ? 4 : K <= 8 ? 8 : 16; }

constexpr size_t kSmemLimit = 227 * 1024;

// Layout of a launch's shared memory.
struct TcLayout {
    int stages;
    bool alias;
    uint32_t exch_off, win_off, staging_off, tail_off;
    size_t smem;
};

// Shared memory of a launch: 1 KiB alignment slack, the TMA ring, then
// (split mode) the DSMEM staging area, the epilogue exchange area, the tail
// and the bias.  Split CTAs run only kb_per K-steps, so their ring needs no
// more stages than that; they prefer to fit two CTAs per SM.  With alias set
// the staging area overlays the ring instead (it is written only once every
// CTA of the cluster has finished its MMAs), for gates so wide that a ring
// beside it would hold a single stage.
bool layout_for(int EP, int NP, int kmax, bool split, int kb_per, bool alias, TcLayout &L, int nparts = 2,
                int kpack = 1, bool wide = false)
{
    const size_t slot = (kABytes + static_cast<size_t>(EP) * kBK * 2) * kpack;
    const size_t staging = split ? static_cast<size_t>(kBM) * stage_row_floats(NP) * sizeof(float) : 0;
    const size_t apart = alias ? 0 : staging;
    const size_t exch = (split ? 0 : exch_lists_bytes(kmax, nparts)) + win_bytes(kmax);
    const size_t fixed = 1024 + apart + exch + sizeof(TcSmemTail) + (sizeof(float) + sizeof(int)) * EP;
    const int max_st = split ? (kb_per < kMaxStages ? (kb_per < 1 ? 1 : kb_per) : kMaxStages) : kMaxStages;
    const int min_st = split ? 1 : 2;
    const size_t budgets[2] = {split && !wide ? static_cast<size_t>(113 * 1024) : kSmemLimit, kSmemLimit};
    for (size_t budget : budgets) {
        for (int st = max_st; st >= min_st; --st) {
            size_t ring = static_cast<size_t>(st) * slot;
            if (alias && ring < staging) ring = staging;
            ring = (ring + 1023) & ~size_t(1023);
            if (fixed + ring <= budget) {
                L.stages = st;
                L.alias = alias && split;
                L.staging_off = static_cast<uint32_t>(alias ? 0 : ring);
                L.exch_off = static_cast<uint32_t>(ring + apart);
                L.win_off = static_cast<uint32_t>(ring + apart + (split ? 0 : exch_lists_bytes(kmax, nparts)));
                L.tail_off = static_cast<uint32_t>(ring + apart + exch);
                L.smem = fixed + ring;
                return true;
            }
        }
    }
    return false;
}

// Split-mode layout: the staging area apart from the ring unless that leaves
// a one-stage ring for more than one K-step and the overlay does better.
bool split_layout(int EP, int NP, int kmax, int kb_per, TcLayout &L, bool wide = false)
{
    const bool ok = layout_for(EP, NP, kmax, true, kb_per, false, L, 2, 1, wide);
    if (ok && (L.stages > 1 || kb_per <= 1)) return true;
    TcLayout A;
    if (layout_for(EP, NP, kmax, true, kb_per, true, A, 2, 1, wide) && (!ok || A.stages > L.stages)) {
        L = A;
        return true;
    }
    return ok;
}

template <int KMAX, bool SPLIT, bool FUSE = false>
cudaError_t set_smem_attr(int dev)
{
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev & 63);
    if (configured.load() & bit) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(route_tc_kernel<KMAX, SPLIT, FUSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSmemLimit));
    if (err == cudaSuccess) configured.fetch_or(bit);
    return err;
}

template <int KMAX, bool FUSE = false>
int max_active_clusters(size_t smem, int S, int dev)
{
    // cached per (device, cluster size, shared memory size)
    static std::mutex mu;
    static std::map<uint64_t, int> cache;
    const uint64_t key = (static_cast<uint64_t>(KMAX) << 52) | (static_cast<uint64_t>(FUSE) << 48) |
                         (static_cast<uint64_t>(dev) << 40) | (static_cast<uint64_t>(S) << 32) | smem;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, route_tc_kernel<KMAX, true, FUSE>, &cfg) != cudaSuccess) n = 0;
    std::lock_guard<std::mutex> g(mu);
    cache[key] = n;
    return n;
}

template <int KMAX>
cudaError_t plan_and_launch(const RouteArgs &a, const CUtensorMap &tmX, const CUtensorMap &tmW, cudaStream_t stream,
                            int dev, const FuseArgs *fz = nullptr)
{
    const int sms = device_sm_count(dev);
    TcParams q;
    q.bias = a.bias;
    q.topk_idx = a.topk_idx;
    q.topk_w = a.topk_w;
    q.status = a.status;
    q.lse = a.lse;
    q.counts = a.counts;
    q.d_counts = fz ? fz->counts : nullptr;
    q.d_offsets = fz ? fz->offsets : nullptr;
    q.d_row_map = fz ? fz->row_map : nullptr;
    q.d_src_slot = fz ? fz->src_slot : nullptr;
    q.d_X = static_cast<const uint4 *>(a.X);
    q.d_Xp = fz ? static_cast<uint4 *>(fz->X_perm) : nullptr;
    q.d_bar = fz ? static_cast<unsigned *>(fz->workspace) : nullptr;
    q.d_hist = fz ? reinterpret_cast<int32_t *>(static_cast<unsigned char *>(fz->workspace) + 256) : nullptr;
    q.N = static_cast<int>(a.N);
    q.H = a.H;
    q.E = a.E;
    q.K = a.K;
    q.renorm = a.renorm;
    q.need_z = (!a.renorm || a.lse != nullptr) ? 1 : 0;
    q.EP = (a.E + 63) / 64 * 64;
    q.NP = (a.E + 15) / 16 * 16;
    q.tiles = static_cast<int>((a.N + kBM - 1) / kBM);
    q.kpack = 1;
    q.x_keep = keep_in_l2(a.N * 2 * static_cast<int64_t>(a.H), dev) ? 1 : 0;
    const int nk = (a.H + kBK - 1) / kBK;

    // split H over a cluster while the tiles alone leave SMs idle
    int S = 1;
    while (S < 8 && static_cast<int64_t>(q.tiles) * S * 2 <= sms && nk >= 2 * S) S *= 2;

    cudaError_t err;
    TcLayout L;
    if (S > 1) {
        if ((err = fz ? set_smem_attr<KMAX, true, true>(dev) : set_smem_attr<KMAX, true>(dev)) != cudaSuccess)
            return err;
        // every cluster must be resident at once (one wave), else use a smaller split
        for (; S > 1; S >>= 1) {
            if (!split_layout(q.EP, q.NP, KMAX, (nk + S - 1) / S, L)) continue;
            const int fit = fz ? max_active_clusters<KMAX, true>(L.smem, S, dev)
                               : max_active_clusters<KMAX>(L.smem, S, dev);
            if (fit >= q.tiles) break;
        }
    }
    const bool split = S > 1;
    // route + dispatch in one launch needs the split mode (one wave of CTAs); a
    // large row copy is left to the dispatch kernel, which spreads it over every SM
    if (fz && (!split || static_cast<int64_t>(S) * q.tiles > kFuseMaxCtas ||
               (fz->X_perm != nullptr && a.N * a.K * 2 * static_cast<int64_t>(a.H) > kFuseMaxCopyBytes)))
        return cudaErrorNotSupported;
    // persistent mode: tiles of fewer than kBM tokens where that lets every SM
    // take the same number of tiles (each still loads a kBM-row box; the rows
    // past its own are the next tile's, read from L2 a second time)
    q.tile_rows = kBM;
    if (!split) {
        const int64_t waves = (q.tiles + sms - 1) / sms;
        const int64_t rows = (a.N + waves * sms - 1) / (waves * sms);
        if (rows >= 8 && rows < kBM) {
            q.tile_rows = static_cast<int>(rows);
            q.tiles = static_cast<int>((a.N + rows - 1) / rows);
        }
    }
    // persistent mode: two K-steps per ring stage where the 3D view of X can be
    // encoded (one X copy and one gate-weight copy per 64 experts bring 32 KiB of X).
    // MOE_ROUTE_KPACK=1 (read once per process) keeps one K-step per stage.
    CUtensorMap tmX3, tmW2;
    static const bool kpack1 = [] {
        const char *v = std::getenv("MOE_ROUTE_KPACK");
        return v != nullptr && std::strcmp(v, "1") == 0;
    }();
    if (!split && !kpack1 && encode_x_3d(&tmX3, a.X, static_cast<uint64_t>(a.H), static_cast<uint64_t>(a.N), kBM) &&
        encode_2d_bf16(&tmW2, a.W, static_cast<uint64_t>(a.E), static_cast<uint64_t>(a.H), 64, 2 * kBK) &&
        layout_for(q.EP, q.NP, KMAX, false, nk, false, L, TcShape<KMAX, false>::kParts, 2) && L.stages >= 3)
        q.kpack = 2;
    if (q.kpack == 1 && (split ? !split_layout(q.EP, q.NP, KMAX, (nk + S - 1) / S, L)
                               : !layout_for(q.EP, q.NP, KMAX, false, nk, false, L, TcShape<KMAX, false>::kParts)))
        return cudaErrorInvalidConfiguration;
    // route + dispatch with one CTA per SM: the layout may take the whole of shared
    // memory, so that the CTA's rows of X fit beside the dispatch scratch and leave
    // as bulk stores (the planned clusters must still all be resident at once)
    if (fz && split && fz->X_perm != nullptr && static_cast<int64_t>(S) * q.tiles <= sms) {
        TcLayout W;
        if (split_layout(q.EP, q.NP, KMAX, (nk + S - 1) / S, W, true) && W.smem > L.smem &&
            max_active_clusters<KMAX, true>(W.smem, S, dev) >= q.tiles)
            L = W;
    }
    q.stages = L.stages;
    q.exch_off = L.exch_off;
    q.win_off = L.win_off;
    q.staging_off = L.staging_off;
    q.tail_off = L.tail_off;
    q.staging_alias = L.alias ? 1 : 0;
    q.nsplit = S;
    q.d_prefetch = 0;
    q.d_scr_off = L.staging_off;
    if (fz) {
        // the dispatch scratch: an mbarrier (16 bytes) and the counts; with room,
        // the CTA's kBM / S rows of X are first copied to offset 0 of shared memory
        const size_t R = static_cast<size_t>(kBM / S);
        const size_t scratch = 16 + sizeof(int) * (13 * static_cast<size_t>(a.E) + 2 + R * a.K);
        const size_t rows_bytes = (R * 2 * a.H + 15) & ~size_t(15);
        if (fz->X_perm != nullptr && rows_bytes + scratch <= L.tail_off) {
            q.d_prefetch = 1;
            q.d_scr_off = static_cast<uint32_t>(rows_bytes);
        }
    }
    q.kb_per = (nk + S - 1) / S;
    uint32_t cols = 32;
    const uint32_t need = static_cast<uint32_t>(split ? q.NP : 2 * q.NP);  // persistent: two accumulators
    while (cols < need) cols <<= 1;
    q.tmem_cols = cols;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[3];
    int na = 0;
    if (split) {
        cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(q.tiles), 1);
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = S;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    } else {
        cfg.gridDim = dim3(static_cast<unsigned>(q.tiles < sms ? q.tiles : sms), 1, 1);
    }
    cfg.blockDim = dim3(static_cast<unsigned>(split ? TcShape<KMAX, true>::kThr : TcShape<KMAX, false>::kThr), 1, 1);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (fz) {
        // all CTAs resident at once: the grid barrier of the dispatch part cannot
        // deadlock.  MOE_FUSED_LAUNCH (read once per process) changes the launch:
        //  "noncooperative": without the cooperative attribute (profilers run
        //      cooperative cluster launches without clusters; a plain cluster launch
        //      keeps them); the one-wave check above still places every CTA at once
        //      on an idle GPU;
        //  "nocluster": cooperative but without the cluster dimension, so that every
        //      CTA runs the kernel's solo branch, as under such a profiler (a test
        //      switch for that branch).
        static const int mode = [] {
            const char *v = std::getenv("MOE_FUSED_LAUNCH");
            if (v != nullptr && std::strcmp(v, "noncooperative") == 0) return 1;
            if (v != nullptr && std::strcmp(v, "nocluster") == 0) return 2;
            return 0;
        }();
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        cfg.numAttrs = mode == 1 ? na : na + 1;
        if (mode == 2) {   // drop the cluster dimension (attr[0])
            cfg.attrs = attr + 1;
            cfg.numAttrs = na;
        }
        err = cudaLaunchKernelEx(&cfg, route_tc_kernel<KMAX, true, true>, tmX, tmW, q);
        if (err != cudaSuccess) {
            (void)cudaGetLastError();   // not launched: the caller routes and dispatches apart
            return cudaErrorNotSupported;
        }
        return cudaSuccess;
    }
    if (split) return cudaLaunchKernelEx(&cfg, route_tc_kernel<KMAX, true>, tmX, tmW, q);
    if ((err = set_smem_attr<KMAX, false>(dev)) != cudaSuccess) return err;
    if (q.kpack == 2) return cudaLaunchKernelEx(&cfg, route_tc_kernel<KMAX, false>, tmX3, tmW2, q);
    return cudaLaunchKernelEx(&cfg, route_tc_kernel<KMAX, false>, tmX, tmW, q);
}

}  // namespace

bool route_tc_supported(const RouteArgs &a, int device)
{
    if (device_cc_major(device) != 10) return false;  // tcgen05: sm_100 family
    if (a.E % 8 != 0 || a.E > 256) return false;      // gate rows must be 16-byte multiples for TMA
    if (a.H % 8 != 0) return false;
    if (a.N > 0x7fffffff - kBM) return false;
    if (reinterpret_cast<uintptr_t>(a.X) % 16 || reinterpret_cast<uintptr_t>(a.W) % 16) return false;
    return encode_tiled_fn() != nullptr;
}

cudaError_t launch_route_dispatch_tc(const RouteArgs &a, const FuseArgs &f, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (!route_tc_supported(a, dev)) return cudaErrorNotSupported;
    CUtensorMap tmX, tmW;
    if (!encode_2d_bf16(&tmX, a.X, static_cast<uint64_t>(a.H), static_cast<uint64_t>(a.N), kBK, kBM))
        return cudaErrorInvalidValue;
    if (!encode_2d_bf16(&tmW, a.W, static_cast<uint64_t>(a.E), static_cast<uint64_t>(a.H), 64, kBK))
        return cudaErrorInvalidValue;
    switch (kmax_for(a.K)) {
    case 2: return plan_and_launch<2>(a, tmX, tmW, stream, dev, &f);
    case 4: return plan_and_launch<4>(a, tmX, tmW, stream, dev, &f);
    case 8: return plan_and_launch<8>(a, tmX, tmW, stream, dev, &f);
    default: return plan_and_launch<16>(a, tmX, tmW, stream, dev, &f);
    }
}

cudaError_t launch_route_tc(const RouteArgs &a, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    CUtensorMap tmX, tmW;
    if (!encode_2d_bf16(&tmX, a.X, static_cast<uint64_t>(a.H), static_cast<uint64_t>(a.N), kBK, kBM))
        return cudaErrorInvalidValue;
    if (!encode_2d_bf16(&tmW, a.W, static_cast<uint64_t>(a.E), static_cast<uint64_t>(a.H), 64, kBK))
        return cudaErrorInvalidValue;
    switch (kmax_for(a.K)) {
    case 2: return plan_and_launch<2>(a, tmX, tmW, stream, dev);
    case 4: return plan_and_launch<4>(a, tmX, tmW, stream, dev);
    case 8: return plan_and_launch<8>(a, tmX, tmW, stream, dev);
    default: return plan_and_launch<16>(a, tmX, tmW, stream, dev);
    }
}

}  // namespace moe
