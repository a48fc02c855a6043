// dispatch.cu -- counting-sort dispatch metadata and the row permute.
//
// The PithTrain page ("一万行Python构建MoE训练栈：解构4D并行、DualPipeV调度与FP8算子",
// §8.2 O(n) counting sort 替代 O(n log n) argsort) builds the dispatch in
// three kernels: a bincount with per-CTA private histograms, a one-CTA
// reduction + prefix sum, and a scatter that writes expand_idx.  On GB300 the
// three phases fit in ONE launch of a thread-block cluster (up to 8 CTAs of
// 1024 threads): each CTA histograms its contiguous range of slots in shared
// memory, the cluster barrier publishes the per-CTA histograms, every CTA
// reads its peers' histograms through distributed shared memory to get its
// base row per expert, and then scatters.  No global workspace, no global
// atomics, no inter-CTA spin waits.
//
// Ordering: rows are ordered by (expert, slot), slot = n*K + k.  Within a
// CTA, warp w owns a contiguous sub-range of slots and walks it 32 slots at a
// time; ballots on the bits of the expert id group equal experts of a step and
// the rank inside the group (lanes below) keeps slot order.
#include <atomic>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMetaThreads = 1024;
constexpr int kMetaWarps = kMetaThreads / 32;
constexpr int kMaxE = 256;
constexpr int kMaxCluster = 8;
constexpr size_t kMetaSmemMax = 200 * 1024;  // dynamic shared memory of the metadata kernel

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ int ld_dsmem_i32(const int *local_ptr, uint32_t cta)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_ptr)), "r"(cta));
    int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

// Shared memory of the metadata kernel.
struct MetaSmem {
    int cta_hist[kMaxE];   // this CTA's count per expert (read by peers)
    int total[kMaxE];      // cluster-wide count per expert
    int before[kMaxE];     // counts of lower-ranked CTAs
    int offset[kMaxE + 1]; // exclusive prefix of total
    int bad;               // an out-of-range index was seen
    // followed by: int wcnt[kMetaWarps][E], then uint16 stage[stage_cap]
};

constexpr uint16_t kInvalid = 0xFFFFu;
constexpr uint16_t kIgnore = 0xFFFEu;   // a slot that takes no row and is not an error

// The CTA's slots are first copied into shared memory as 16-bit expert ids
// (0xFFFF marks an id outside [0,E)) with every load in flight at once; both
// passes then read shared memory only.  Slots beyond `stage_cap` (very large
// N*K) are read from global memory in the passes instead.
__device__ __forceinline__ int slot_expert(const uint16_t *stage, int64_t c0, int64_t staged_end,
                                           const int32_t *__restrict__ topk_idx, int64_t s, int E)
{
    if (s < staged_end) {
        const uint16_t v = stage[s - c0];
        return v == kInvalid ? -1 : static_cast<int>(v);
    }
    const int e = topk_idx[s];
    return (e < 0 || e >= E) ? -1 : e;
}

__global__ void __launch_bounds__(kMetaThreads, 1) dispatch_meta_kernel(
    const int32_t *__restrict__ topk_idx, int64_t S, int E, int stage_cap, int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ row_map, int32_t *__restrict__ src_slot,
    int32_t *status)
{
    extern __shared__ __align__(16) unsigned char meta_raw[];
    MetaSmem &sm = *reinterpret_cast<MetaSmem *>(meta_raw);
    int *wcnt = reinterpret_cast<int *>(meta_raw + sizeof(MetaSmem));
    uint16_t *stage = reinterpret_cast<uint16_t *>(wcnt + kMetaWarps * E);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t nctas = cluster_nctarank();

    // Slot ranges: CTA rank gets [c0, c1), warp w gets [w0, w1) inside it.
    const int64_t per_cta = (S + nctas - 1) / nctas;
    const int64_t c0 = min(S, per_cta * rank);
    const int64_t c1 = min(S, c0 + per_cta);
    const int64_t staged_end = min(c1, c0 + static_cast<int64_t>(stage_cap));
    const int64_t per_warp = (c1 - c0 + kMetaWarps - 1) / kMetaWarps;
    const int64_t w0 = min(c1, c0 + per_warp * warp);
    const int64_t w1 = min(c1, w0 + per_warp);
    int *my_cnt = wcnt + warp * E;

    for (int i = tid; i < kMetaWarps * E; i += kMetaThreads) wcnt[i] = 0;
    if (tid == 0) sm.bad = 0;
    __syncthreads();

    // a single cluster: the next kernel may start launching now (it still
    // waits for this grid to complete)
    pdl_launch_dependents();
    pdl_wait_prior_grids();

    // ---- stage the CTA's expert ids (independent loads, unrolled)
    bool bad = false;
    const int nst = static_cast<int>(staged_end - c0);
#pragma unroll 8
    for (int i = tid; i < nst; i += kMetaThreads) {
        const int e = topk_idx[c0 + i];
        const bool ok = e >= 0 && e < E;
        bad |= !ok;
        stage[i] = ok ? static_cast<uint16_t>(e) : kInvalid;
    }
    for (int64_t s = staged_end + tid; s < c1; s += kMetaThreads) {
        const int e = topk_idx[s];
        bad |= !(e >= 0 && e < E);
    }
    if (bad) sm.bad = 1;
    __syncthreads();

    // ---- phase 1: per-warp histograms of the warp's slots
    // (ids outside [0,E) and lanes past the end share the key E, which is never counted)
    for (int64_t base = w0; base < w1; base += 32) {
        const int64_t s = base + lane;
        int e = s < w1 ? slot_expert(stage, c0, staged_end, topk_idx, s, E) : -1;
        if (e < 0) e = E;
        const uint32_t peers = same_key_lanes(e);
        if (e < E && lane == __ffs(peers) - 1) my_cnt[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // ---- CTA totals; per-warp exclusive prefix (in place)
    for (int e = tid; e < E; e += kMetaThreads) {
        int run = 0;
        for (int w = 0; w < kMetaWarps; ++w) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
        sm.cta_hist[e] = run;
    }
    cluster_arrive_release();
    cluster_wait_acquire();

    // ---- read every CTA's histogram through distributed shared memory
    for (int e = tid; e < E; e += kMetaThreads) {
        int tot = 0, bef = 0;
        for (uint32_t c = 0; c < nctas; ++c) {
            const int v = ld_dsmem_i32(&sm.cta_hist[e], c);
            tot += v;
            if (c < rank) bef += v;
        }
        sm.total[e] = tot;
        sm.before[e] = bef;
    }
    // Peers may leave once everyone has finished reading: arrive now, wait at the end.
    cluster_arrive_release();
    __syncthreads();

    // ---- exclusive scan over experts (E <= 256: one warp, 8 per lane)
    if (warp == 0) {
        int vals[kMaxE / 32];
        int local = 0;
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i) {
            const int e = lane * (kMaxE / 32) + i;
            vals[i] = e < E ? sm.total[e] : 0;
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
        for (int i = 0; i < kMaxE / 32; ++i) {
            const int e = lane * (kMaxE / 32) + i;
            if (e < E) sm.offset[e] = run;
            run += vals[i];
        }
        if (lane == 31) sm.offset[E] = incl;
    }
    __syncthreads();

    if (rank == 0) {
        for (int e = tid; e <= E; e += kMetaThreads) {
            offsets[e] = sm.offset[e];
            if (e < E) counts[e] = sm.total[e];
        }
    }
    for (int i = tid; i < kMetaWarps * E; i += kMetaThreads) {
        const int e = i % E;
        wcnt[i] += sm.offset[e] + sm.before[e];
    }
    __syncthreads();

    // ---- phase 2: stable scatter
    for (int64_t base = w0; base < w1; base += 32) {
        const int64_t s = base + lane;
        int e = s < w1 ? slot_expert(stage, c0, staged_end, topk_idx, s, E) : -1;
        if (e < 0) e = E;
        const uint32_t peers = same_key_lanes(e);
        const uint32_t below = peers & ((1u << lane) - 1u);
        if (s < w1) {
            if (e < E) {
                const int r = my_cnt[e] + __popc(below);
                row_map[s] = r;
                if (src_slot) src_slot[r] = static_cast<int32_t>(s);
            } else {
                row_map[s] = -1;
            }
        }
        __syncwarp();
        if (e < E && below == 0) my_cnt[e] += __popc(peers);
        __syncwarp();
    }

    if (sm.bad && tid == 0) report_status(status, MOE_ERR_BAD_INDEX);
    cluster_wait_acquire();
}

// ---------------------------------------------------------------------------
// Permute (+ E4M3 1x128 block quantisation)
// ---------------------------------------------------------------------------
constexpr int kPermWarps = 8;

// fl32(1/448): 1/448 = (8/7) * 2^-9 rounded to nearest binary32.
constexpr uint32_t kRcp448Bits = 0x3B124925u;

__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Block-scale output: fp32 scales, or UE8M0 bytes (biased exponent, scale =
// 2^(byte - 127)) -- the fp32 and e8m0 branches of the quantiser (PithTrain
// page, §7.2 架构感知的量化核, _compute_fp8_scale).
struct ScaleOut {
    void *ptr;   // float [rows, H/128] or uint8 [rows, H/128]
    int ue8m0;
};

// Quantise 8 bf16 values (one 16-byte chunk) held by each lane; lanes 0-15 and
// 16-31 each hold one 128-element block.  Returns the 8 E4M3 codes and the
// block's power-of-two scale s (x ~ q * s).  Both branches take the same fp32
// product t; the fp32 branch raises t to a power of two by its bit rule, the
// e8m0 branch by the hardware round-toward-+inf conversion to UE8M0 (the same
// value for every positive finite t).
__device__ __forceinline__ uint2 quant_chunk_e4m3(const uint4 &x, float &s_out, int ue8m0)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    float f[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        f[2 * p] = __uint_as_float(w[p] << 16);
        f[2 * p + 1] = __uint_as_float(w[p] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int p = 0; p < 8; ++p) amax = fmaxf(amax, fabsf(f[p]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // t = fl32(max(amax, 1e-4) * fl32(1/448)); s = t's exponent, bumped when t has a non-zero mantissa
    const float t = __fmul_rn(fmaxf(amax, 1e-4f), __uint_as_float(kRcp448Bits));
    uint32_t sbits;
    if (ue8m0) {
        uint16_t e;
        asm("cvt.rp.satfinite.ue8m0x2.f32 %0, %1, %2;" : "=h"(e) : "f"(0.0f), "f"(t));
        sbits = static_cast<uint32_t>(e & 0xFFu) << 23;
    } else {
        const uint32_t tb = __float_as_uint(t);
        sbits = (tb & 0x7F800000u) + ((tb & 0x007FFFFFu) ? 0x00800000u : 0u);
    }
    s_out = __uint_as_float(sbits);
    const float inv_s = __uint_as_float((254u - (sbits >> 23)) << 23);  // exact 1/s (a power of two)
    uint2 q;
    q.x = f32x2_to_e4m3x2(f[0] * inv_s, f[1] * inv_s) | (f32x2_to_e4m3x2(f[2] * inv_s, f[3] * inv_s) << 16);
    q.y = f32x2_to_e4m3x2(f[4] * inv_s, f[5] * inv_s) | (f32x2_to_e4m3x2(f[6] * inv_s, f[7] * inv_s) << 16);
    return q;
}

// Copy one token's row to its K destination rows (and/or quantise it), one
// warp.  Lane k < K holds the destination row of slot k in `my_row` (-1: skip).
// A lane holds CPL 16-byte chunks of the row at once (chunk base + lane + 32 j),
// so a whole row slice is in flight before any store; rows wider than
// 32 * CPL chunks take several batches.
template <int CPL>
__device__ __forceinline__ void load_row_batch(const uint4 *__restrict__ src, int base, int chunks, int lane,
                                               uint4 (&x)[CPL])
{
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const int c = base + lane + 32 * j;
        x[j] = c < chunks ? __ldcs(src + c) : make_uint4(0, 0, 0, 0);
    }
}

template <bool kFp8, int CPL>
__device__ __forceinline__ void quant_row_batch(const uint4 (&x)[CPL], uint2 (&q)[kFp8 ? CPL : 1],
                                                float (&sc)[kFp8 ? CPL : 1], int ue8m0)
{
    if constexpr (kFp8) {
#pragma unroll
        for (int j = 0; j < CPL; ++j) q[j] = quant_chunk_e4m3(x[j], sc[j], ue8m0);
    }
}

// Row stores: streamed through L2 (evict-first), or, where the whole output
// fits in L2 next to what is still in use (`keep`), with the default
// write-back policy, so that the kernel that reads the rows next finds them there.
template <typename T>
__device__ __forceinline__ void st_row(T *p, const T &v, int keep)
{
    if (keep)
        *p = v;
    else
        __stcs(p, v);
}

template <bool kBf16Out, bool kFp8, int CPL>
__device__ __forceinline__ void store_row_batch(const uint4 (&x)[CPL], const uint2 (&q)[kFp8 ? CPL : 1],
                                                const float (&sc)[kFp8 ? CPL : 1], int base, int my_row, int K,
                                                int H, uint4 *__restrict__ Xp, uint8_t *__restrict__ Xq,
                                                const ScaleOut Xs, int lane, int keep)
{
    const int chunks = H >> 3;
    const int nb = H >> 7;
    for (int k = 0; k < K; ++k) {
        const int r = __shfl_sync(0xffffffffu, my_row, k);
        if (r < 0) continue;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = base + lane + 32 * j;
            if (c >= chunks) continue;
            if constexpr (kBf16Out) st_row(Xp + static_cast<int64_t>(r) * chunks + c, x[j], keep);
            if constexpr (kFp8) {
                st_row(reinterpret_cast<uint2 *>(Xq + static_cast<int64_t>(r) * H) + c, q[j], keep);
                if ((lane & 15) == 0) {
                    const int64_t at = static_cast<int64_t>(r) * nb + (c >> 4);
                    if (Xs.ue8m0)
                        static_cast<uint8_t *>(Xs.ptr)[at] = static_cast<uint8_t>(__float_as_uint(sc[j]) >> 23);
                    else
                        static_cast<float *>(Xs.ptr)[at] = sc[j];
                }
            }
        }
    }
}

// Copy one token's row to its K destination rows (and/or quantise it), one
// warp.  Lane k < K holds the destination row of slot k in `my_row` (-1: skip).
// A lane holds CPL 16-byte chunks of the row at once (chunk base + lane + 32 j),
// so a whole row slice is in flight before any store; rows wider than
// 32 * CPL chunks take several batches.
template <bool kBf16Out, bool kFp8, int CPL>
__device__ __forceinline__ void copy_token_rows(const uint4 *__restrict__ src, int my_row, int K, int H,
                                                uint4 *__restrict__ Xp, uint8_t *__restrict__ Xq,
                                                const ScaleOut Xs, int lane, int keep)
{
    const int chunks = H >> 3;  // 16-byte chunks per row
    for (int base = 0; base < chunks; base += 32 * CPL) {
        uint4 x[CPL];
        uint2 q[kFp8 ? CPL : 1];
        float sc[kFp8 ? CPL : 1];
        load_row_batch<CPL>(src, base, chunks, lane, x);
        quant_row_batch<kFp8, CPL>(x, q, sc, Xs.ue8m0);
        store_row_batch<kBf16Out, kFp8, CPL>(x, q, sc, base, my_row, K, H, Xp, Xq, Xs, lane, keep);
    }
}

template <bool kBf16Out, bool kFp8, int CPL>
__global__ void __launch_bounds__(kPermWarps * 32) permute_kernel(
    const uint4 *__restrict__ X, const int32_t *__restrict__ row_map, int64_t N, int H, int K,
    uint4 *__restrict__ Xp, uint8_t *__restrict__ Xq, const ScaleOut Xs, int32_t *status, int skip_unset, int keep)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rows = N * K;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kPermWarps;

    pdl_wait_prior_grids();

    bool bad = false;
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * kPermWarps + warp; n < N; n += nwarps) {
        int my_row = -1;
        if (lane < K) {
            my_row = row_map[n * K + lane];
            if (my_row < 0 || my_row >= rows) {
                bad |= !(skip_unset && my_row == -1);  // -1: a slot that takes no row, when allowed
                my_row = -1;
            }
        }
        copy_token_rows<kBf16Out, kFp8, CPL>(X + n * (H >> 3), my_row, K, H, Xp, Xq, Xs, lane, keep);
    }
    if (bad) report_status(status, MOE_ERR_BAD_INDEX);
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Fused dispatch: counting sort + permute in ONE cooperative launch
// ---------------------------------------------------------------------------
// One CTA per SM (all resident: cooperative launch).  CTA c owns a contiguous
// token range.  Phase 1: the CTA's expert ids are staged in shared memory and
// counted per warp (per-warp histograms, ballot-grouped); the CTA's counts go
// to a small global workspace.  A bounded grid barrier follows.  Phase 2: every
// CTA reads all CTAs' counts from L2, forms expert_offsets and its own base row
// per expert, scatters row_map / src_slot in (expert, slot) order, and copies
// its tokens' rows to their destinations (+ E4M3) right away.  The barrier
// counters live in the workspace: they must be zero before the first call and
// the last CTA to leave returns them to zero.
constexpr int kFusedThreads = 512;
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedMaxSlots = 16384;   // slots per CTA staged in shared memory
constexpr int kFusedMaxCtas = 1024;     // bound used to size the workspace
constexpr int kHistBatch = 32;          // per-thread count loads in flight at once
constexpr int kHistBatch4 = 8;          // the same for 16-byte loads of four counts

struct FusedParams {
    const int32_t *topk_idx;
    const uint4 *X;
    int64_t N;
    int H, E, K;
    int tok_per;   // tokens per CTA
    int32_t *counts, *offsets, *row_map, *src_slot;
    uint4 *Xp;
    uint8_t *Xq;
    ScaleOut Xs;
    int32_t *status;
    unsigned *bar;  // [0] arrive, [1] depart
    int32_t *hist;  // [gridDim.x][E]
    int ep_P;       // 0: keys are the expert ids; > 0: keys are EP ranks (E of them, ep_P experts each)
    int keep;       // rows stored with the default write-back policy (they fit in L2), else streamed
};

struct FusedSmem {
    int total[kMaxE];       // grid-wide count per expert
    int before[kMaxE];      // counts of lower CTAs
    int offset[kMaxE + 1];  // exclusive prefix of total
    int bad;
    int ok;
    // followed by: int wcnt[kFusedWarps][E]; int rows[slots]; uint16 stage[slots]
};

template <bool kBf16Out, bool kFp8, int CPL>
__global__ void __launch_bounds__(kFusedThreads, 1) dispatch_fused_kernel(const FusedParams p)
{
    extern __shared__ __align__(16) unsigned char fz_raw[];
    FusedSmem &sm = *reinterpret_cast<FusedSmem *>(fz_raw);
    const int E = p.E;
    const int K = p.K;
    int *wcnt = reinterpret_cast<int *>(fz_raw + sizeof(FusedSmem));
    int *rows_s = wcnt + kFusedWarps * E;
    uint16_t *stage = reinterpret_cast<uint16_t *>(rows_s + p.tok_per * K);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int c = blockIdx.x;
    const unsigned G = gridDim.x;
    const int64_t t0 = min(p.N, static_cast<int64_t>(c) * p.tok_per);
    const int64_t t1 = min(p.N, t0 + p.tok_per);
    const int64_t s0 = t0 * K;
    const int ns = static_cast<int>((t1 - t0) * K);   // slots of this CTA
    const int per_warp = (ns + kFusedWarps - 1) / kFusedWarps;
    const int w0 = min(ns, per_warp * warp);
    const int w1 = min(ns, w0 + per_warp);
    int *my_cnt = wcnt + warp * E;

    for (int i = tid; i < kFusedWarps * E; i += kFusedThreads) wcnt[i] = 0;
    for (int e = tid; e < E; e += kFusedThreads) {
        sm.total[e] = 0;
        sm.before[e] = 0;
    }
    if (tid == 0) sm.bad = 0;
    __syncthreads();

    // One wave of CTAs (cooperative launch): the next kernel may start
    // launching now; it still waits for this grid to complete.
    pdl_launch_dependents();
    pdl_wait_prior_grids();

    // ---- each warp's first token row does not depend on the metadata: load
    // (and quantise) it now, so its latency hides behind the counting phases
    const int ntok = static_cast<int>(t1 - t0);
    const int chunks = p.H >> 3;
    const bool pre = (kBf16Out || kFp8) && warp < ntok && chunks <= 32 * CPL;
    uint4 xpre[CPL];
    uint2 qpre[kFp8 ? CPL : 1];
    float spre[kFp8 ? CPL : 1];
    if (pre) {
        load_row_batch<CPL>(p.X + (t0 + warp) * chunks, 0, chunks, lane, xpre);
        quant_row_batch<kFp8, CPL>(xpre, qpre, spre, p.Xs.ue8m0);
    }

    // ---- stage the CTA's keys (0xFFFF: out of range)
    bool bad = false;
    if (p.ep_P == 0) {
#pragma unroll 4
        for (int i = tid; i < ns; i += kFusedThreads) {
            const int e = p.topk_idx[s0 + i];
            const bool ok = e >= 0 && e < E;
            bad |= !ok;
            stage[i] = ok ? static_cast<uint16_t>(e) : kInvalid;
        }
    } else {
        // EP ranks with deduplication: a slot's key is the rank of its expert if no
        // earlier slot of the same token goes to that rank, else it is ignored (no row)
        const int P = p.ep_P;
        for (int i = tid; i < ns; i += kFusedThreads) {
            const int e = p.topk_idx[s0 + i];
            const bool ok = e >= 0 && e < E * P;
            bad |= !ok;
            const int k = i % K;  // CTA slot ranges start at token boundaries
            bool first = true;
            for (int j = i - k; j < i; ++j) {
                const int ej = p.topk_idx[s0 + j];
                first &= !(ej >= 0 && ej < E * P && ej / P == e / P);
            }
            stage[i] = !ok ? kInvalid : first ? static_cast<uint16_t>(e / P) : kIgnore;
        }
    }
    if (bad) sm.bad = 1;
    __syncthreads();

    // ---- phase 1: per-warp histograms (ids outside [0,E) share the key E, never counted)
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        int e = i < w1 ? static_cast<int>(stage[i]) : E;
        if (e >= E) e = E;
        const uint32_t peers = same_key_lanes(e);
        if (e < E && lane == __ffs(peers) - 1) my_cnt[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // CTA count per expert to the workspace; per-warp exclusive prefix in place
    for (int e = tid; e < E; e += kFusedThreads) {
        int run = 0;
        for (int w = 0; w < kFusedWarps; ++w) {
            const int v = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += v;
        }
        p.hist[static_cast<int64_t>(c) * E + e] = run;
    }

    // ---- grid barrier (bounded)
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        red_add_release_gpu(&p.bar[0], 1u);
        const uint64_t tb = globaltimer_ns();
        int ok = 1;
        for (uint32_t it = 0; ld_acquire_gpu(&p.bar[0]) < G; ++it) {
            if ((it & 255u) == 255u && globaltimer_ns() - tb > kWaitLimitNs) {
                ok = 0;
                break;
            }
        }
        sm.ok = ok;
    }
    __syncthreads();
    if (!sm.ok) {
        if (tid == 0) report_status(p.status, MOE_ERR_TIMEOUT);
        return;
    }

    // ---- phase 2: grid-wide counts and this CTA's base rows (all CTAs' counts from L2).
    // Thread (grp, e) sums rows grp, grp + groups, ... of column e; all of its
    // loads are issued before the first add (one L2 round trip), then the
    // per-group partials meet in shared memory.
    if (E % 4 == 0) {
        // four experts per 16-byte load: a quarter of the requests
        const int E4 = E >> 2;
        const int groups = kFusedThreads / E4;  // >= 8 (E <= 256)
        const int e4 = tid % E4;
        const int grp = tid / E4;
        int4 tot = make_int4(0, 0, 0, 0), bef = make_int4(0, 0, 0, 0);
        if (grp < groups) {
            const int4 *h4 = reinterpret_cast<const int4 *>(p.hist) + e4;
            for (int c0 = grp; c0 < static_cast<int>(G); c0 += kHistBatch4 * groups) {
                int4 v[kHistBatch4];
#pragma unroll
                for (int i = 0; i < kHistBatch4; ++i) {
                    const int cc = c0 + i * groups;
                    v[i] = cc < static_cast<int>(G) ? __ldcg(h4 + static_cast<int64_t>(cc) * E4) : make_int4(0, 0, 0, 0);
                }
#pragma unroll
                for (int i = 0; i < kHistBatch4; ++i) {
                    const bool lower = c0 + i * groups < c;
                    tot.x += v[i].x; tot.y += v[i].y; tot.z += v[i].z; tot.w += v[i].w;
                    bef.x += lower ? v[i].x : 0; bef.y += lower ? v[i].y : 0;
                    bef.z += lower ? v[i].z : 0; bef.w += lower ? v[i].w : 0;
                }
            }
            const int e = 4 * e4;
            atomicAdd(&sm.total[e], tot.x); atomicAdd(&sm.total[e + 1], tot.y);
            atomicAdd(&sm.total[e + 2], tot.z); atomicAdd(&sm.total[e + 3], tot.w);
            atomicAdd(&sm.before[e], bef.x); atomicAdd(&sm.before[e + 1], bef.y);
            atomicAdd(&sm.before[e + 2], bef.z); atomicAdd(&sm.before[e + 3], bef.w);
        }
    } else {
        const int groups = kFusedThreads / E;   // >= 2 (E <= 256)
        const int e = tid % E;
        const int grp = tid / E;
        int tot = 0, bef = 0;
        if (grp < groups) {
            for (int c0 = grp; c0 < static_cast<int>(G); c0 += kHistBatch * groups) {
                int v[kHistBatch];
#pragma unroll
                for (int i = 0; i < kHistBatch; ++i) {
                    const int cc = c0 + i * groups;
                    v[i] = cc < static_cast<int>(G) ? __ldcg(p.hist + static_cast<int64_t>(cc) * E + e) : 0;
                }
#pragma unroll
                for (int i = 0; i < kHistBatch; ++i) {
                    tot += v[i];
                    bef += (c0 + i * groups < c) ? v[i] : 0;
                }
            }
            atomicAdd(&sm.total[e], tot);
            atomicAdd(&sm.before[e], bef);
        }
    }
    __syncthreads();
    if (warp == 0) {
        int vals[kMaxE / 32];
        int local = 0;
#pragma unroll
        for (int i = 0; i < kMaxE / 32; ++i) {
            const int e = lane * (kMaxE / 32) + i;
            vals[i] = e < E ? sm.total[e] : 0;
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
        for (int i = 0; i < kMaxE / 32; ++i) {
            const int e = lane * (kMaxE / 32) + i;
            if (e < E) sm.offset[e] = run;
            run += vals[i];
        }
        if (lane == 31) sm.offset[E] = incl;
    }
    __syncthreads();
    if (c == 0) {
        for (int e = tid; e <= E; e += kFusedThreads) {
            p.offsets[e] = sm.offset[e];
            if (e < E) p.counts[e] = sm.total[e];
        }
    }
    for (int i = tid; i < kFusedWarps * E; i += kFusedThreads) {
        const int e = i % E;
        wcnt[i] += sm.offset[e] + sm.before[e];
    }
    __syncthreads();

    // ---- stable scatter of this CTA's slots
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        int e = i < w1 ? static_cast<int>(stage[i]) : E;
        if (e >= E) e = E;
        const uint32_t peers = same_key_lanes(e);
        const uint32_t below = peers & ((1u << lane) - 1u);
        if (i < w1) {
            const int r = e < E ? my_cnt[e] + __popc(below) : -1;
            rows_s[i] = r;
            p.row_map[s0 + i] = r;
            if (e < E && p.src_slot) p.src_slot[r] = static_cast<int32_t>(s0 + i);
        }
        __syncwarp();
        if (e < E && below == 0) my_cnt[e] += __popc(peers);
        __syncwarp();
    }

    // ---- release the barrier counters (the last CTA to leave resets them)
    if (tid == 0) {
        const unsigned old = atomicAdd(&p.bar[1], 1u);
        if (old == G - 1) {
            p.bar[0] = 0;
            p.bar[1] = 0;
            __threadfence();
        }
    }
    if (sm.bad && tid == 0) report_status(p.status, MOE_ERR_BAD_INDEX);

    // ---- permute this CTA's tokens (rows from shared memory)
    if constexpr (kBf16Out || kFp8) {
        __syncthreads();
        for (int j = warp; j < ntok; j += kFusedWarps) {
            const int my_row = lane < K ? rows_s[j * K + lane] : -1;
            if (j == warp && pre)
                store_row_batch<kBf16Out, kFp8, CPL>(xpre, qpre, spre, 0, my_row, K, p.H, p.Xp, p.Xq, p.Xs, lane,
                                                     p.keep);
            else
                copy_token_rows<kBf16Out, kFp8, CPL>(p.X + (t0 + j) * chunks, my_row, K, p.H, p.Xp, p.Xq, p.Xs,
                                                     lane, p.keep);
        }
    }
}

int meta_cluster_size(int64_t S)
{
    int64_t c = (S + 8191) / 8192;
    if (c < 1) c = 1;
    if (c > kMaxCluster) c = kMaxCluster;
    return static_cast<int>(c);
}

}  // namespace

cudaError_t launch_dispatch_meta(const int32_t *topk_idx, int64_t N, int E, int K, int32_t *counts,
                                 int32_t *offsets, int32_t *row_map, int32_t *src_slot, int32_t *status,
                                 cudaStream_t stream)
{
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        err = cudaFuncSetAttribute(dispatch_meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMetaSmemMax);
        if (err != cudaSuccess) return err;
        configured.fetch_or(bit);
    }
    const int64_t S = N * K;
    const int cl = meta_cluster_size(S);
    const int64_t per_cta = (S + cl - 1) / cl;
    const size_t fixed = sizeof(MetaSmem) + sizeof(int) * kMetaWarps * E;
    const int64_t cap_slots = static_cast<int64_t>((kMetaSmemMax - fixed) / sizeof(uint16_t)) & ~int64_t(7);
    const int stage_cap = static_cast<int>(per_cta < cap_slots ? per_cta : cap_slots);
    const size_t smem = fixed + sizeof(uint16_t) * ((static_cast<size_t>(stage_cap) + 7) & ~size_t(7));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(cl, 1, 1);
    cfg.blockDim = dim3(kMetaThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, dispatch_meta_kernel, topk_idx, S, E, stage_cap, counts, offsets, row_map,
                              src_slot, status);
}

cudaError_t launch_permute(const void *X, const int32_t *row_map, int64_t N, int H, int K, void *X_perm,
                           void *X_fp8, void *X_scale, int scale_ue8m0, int32_t *status, cudaStream_t stream,
                           bool skip_unset)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int sms = device_sm_count(dev);
    const int64_t need = (N + kPermWarps - 1) / kPermWarps;
    const int64_t cap = int64_t(sms) * 8;  // 8 CTAs x 8 warps = 64 warps per SM
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(need < cap ? need : cap), 1, 1);
    cfg.blockDim = dim3(kPermWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint4 *x = static_cast<const uint4 *>(X);
    uint4 *xp = static_cast<uint4 *>(X_perm);
    uint8_t *xq = static_cast<uint8_t *>(X_fp8);
    const ScaleOut xs{X_scale, scale_ue8m0 ? 1 : 0};
    const int chunks = H / 8;
    int cpl = chunks > 256 ? 16 : chunks > 128 ? 8 : chunks > 64 ? 4 : chunks > 32 ? 2 : 1;
    if (X_fp8 && cpl > 8) cpl = 8;  // codes and scales stay live too
    const int64_t out_bytes = N * K * ((X_perm ? 2 * int64_t(H) : 0) + (X_fp8 ? int64_t(H) + H / 32 : 0));
    const int keep = keep_in_l2(out_bytes, dev) ? 1 : 0;
#define MOE_PERMUTE_LAUNCH(B, F, C)                                                            \
    if ((err = prefer_l1_carveout<permute_kernel<B, F, C>>(dev)) != cudaSuccess) return err; \
    return cudaLaunchKernelEx(&cfg, permute_kernel<B, F, C>, x, row_map, N, H, K, xp, xq, xs, status, \
                              skip_unset ? 1 : 0, keep)
#define MOE_PERMUTE_CPL8(B, F)                         \
    switch (cpl) {                                     \
    case 1: MOE_PERMUTE_LAUNCH(B, F, 1);               \
    case 2: MOE_PERMUTE_LAUNCH(B, F, 2);               \
    case 4: MOE_PERMUTE_LAUNCH(B, F, 4);               \
    default: MOE_PERMUTE_LAUNCH(B, F, 8);              \
    }
    if (X_perm && X_fp8) MOE_PERMUTE_CPL8(true, true)
    if (X_fp8) MOE_PERMUTE_CPL8(false, true)
    if (cpl == 16) MOE_PERMUTE_LAUNCH(true, false, 16);
    MOE_PERMUTE_CPL8(true, false)
#undef MOE_PERMUTE_CPL8
#undef MOE_PERMUTE_LAUNCH
}

size_t fused_workspace_bytes(int E) { return 256 + static_cast<size_t>(kFusedMaxCtas) * E * sizeof(int32_t); }

template <bool B, bool F, int C>
cudaError_t launch_fused_t(const FusedParams &p, int grid, size_t smem, cudaStream_t stream, int dev)
{
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev & 63);
    cudaError_t err;
    if (!(configured.load() & bit)) {
        err = cudaFuncSetAttribute(dispatch_fused_kernel<B, F, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   200 * 1024);
        if (err != cudaSuccess) return err;
        configured.fetch_or(bit);
    }
    if ((err = prefer_l1_carveout<dispatch_fused_kernel<B, F, C>>(dev)) != cudaSuccess) return err;
    int occ = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dispatch_fused_kernel<B, F, C>, kFusedThreads, smem);
    if (err != cudaSuccess) return err;
    if (occ < 1 || grid > occ * device_sm_count(dev)) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: the grid barrier cannot deadlock
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, dispatch_fused_kernel<B, F, C>, p);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        cfg.numAttrs = 1;  // without programmatic serialization
        err = cudaLaunchKernelEx(&cfg, dispatch_fused_kernel<B, F, C>, p);
    }
    return err;
}

template <bool B, bool F>
cudaError_t launch_fused_cpl(const FusedParams &p, int grid, size_t smem, cudaStream_t stream, int dev)
{
    const int chunks = p.H / 8;
    // fp8 keeps codes and scales live too: at most 4 chunks per lane (128 registers at 512 threads)
    if constexpr (!F) {
        if (chunks > 128) return launch_fused_t<B, F, 8>(p, grid, smem, stream, dev);
    } else {
        if (chunks > 64) return launch_fused_t<B, F, 4>(p, grid, smem, stream, dev);
    }
    if (chunks > 64) return launch_fused_t<B, F, 4>(p, grid, smem, stream, dev);
    if (chunks > 32) return launch_fused_t<B, F, 2>(p, grid, smem, stream, dev);
    return launch_fused_t<B, F, 1>(p, grid, smem, stream, dev);
}

bool dispatch_fused_supported(int64_t N, int K, int device)
{
    const int sms = device_sm_count(device);
    int64_t grid = sms;
    if (grid > N) grid = N;
    if (grid < 1) return true;
    const int64_t tok_per = (N + grid - 1) / grid;
    grid = (N + tok_per - 1) / tok_per;
    return tok_per * K <= kFusedMaxSlots && grid <= kFusedMaxCtas;
}

cudaError_t launch_dispatch_fused(const int32_t *topk_idx, const void *X, int64_t N, int H, int E, int K,
                                  int32_t *counts, int32_t *offsets, int32_t *row_map, int32_t *src_slot,
                                  void *X_perm, void *X_fp8, void *X_scale, int scale_ue8m0, int32_t *status,
                                  void *workspace, size_t workspace_bytes, cudaStream_t stream, int ep_P)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int sms = device_sm_count(dev);
    int64_t grid = sms;
    if (grid > N) grid = N;
    const int64_t tok_per = (N + grid - 1) / grid;
    grid = (N + tok_per - 1) / tok_per;  // no empty CTAs
    if (tok_per * K > kFusedMaxSlots || grid > kFusedMaxCtas) return cudaErrorNotSupported;
    if (!workspace || workspace_bytes < 256 + static_cast<size_t>(grid) * E * sizeof(int32_t))
        return cudaErrorNotSupported;
    FusedParams p;
    p.topk_idx = topk_idx;
    p.X = static_cast<const uint4 *>(X);
    p.N = N;
    p.H = H;
    p.E = E;
    p.K = K;
    p.tok_per = static_cast<int>(tok_per);
    p.counts = counts;
    p.offsets = offsets;
    p.row_map = row_map;
    p.src_slot = src_slot;
    p.Xp = static_cast<uint4 *>(X_perm);
    p.Xq = static_cast<uint8_t *>(X_fp8);
    p.Xs = ScaleOut{X_scale, scale_ue8m0 ? 1 : 0};
    p.status = status;
    p.bar = static_cast<unsigned *>(workspace);
    p.hist = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) + 256);
    p.ep_P = ep_P;
    p.keep = keep_in_l2(N * K * ((X_perm ? 2 * int64_t(H) : 0) + (X_fp8 ? int64_t(H) + H / 32 : 0)), dev) ? 1 : 0;
    const size_t slots = static_cast<size_t>(tok_per) * K;
    const size_t smem = sizeof(FusedSmem) + sizeof(int) * kFusedWarps * E + sizeof(int) * slots +
                        ((sizeof(uint16_t) * slots + 15) & ~size_t(15));
    const int g = static_cast<int>(grid);
    if (!X) return launch_fused_t<false, false, 1>(p, g, smem, stream, dev);
    if (X_perm && X_fp8) return launch_fused_cpl<true, true>(p, g, smem, stream, dev);
    if (X_fp8) return launch_fused_cpl<false, true>(p, g, smem, stream, dev);
    return launch_fused_cpl<true, false>(p, g, smem, stream, dev);
}

}  // namespace moe
