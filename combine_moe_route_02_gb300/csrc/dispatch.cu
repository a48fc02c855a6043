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
// time; __match_any_sync groups equal experts of a step and the rank inside
// the group (lanes below) keeps slot order.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMetaThreads = 1024;
constexpr int kMetaWarps = kMetaThreads / 32;
constexpr int kMaxE = 256;
constexpr int kMaxCluster = 8;

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
    // followed by: int wcnt[kMetaWarps][E]
};

__global__ void __launch_bounds__(kMetaThreads, 1) dispatch_meta_kernel(
    const int32_t *__restrict__ topk_idx, int64_t S, int E, int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ row_map, int32_t *__restrict__ src_slot,
    int32_t *status)
{
    extern __shared__ __align__(16) unsigned char meta_raw[];
    MetaSmem &sm = *reinterpret_cast<MetaSmem *>(meta_raw);
    int *wcnt = reinterpret_cast<int *>(meta_raw + sizeof(MetaSmem));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t nctas = cluster_nctarank();

    // Slot ranges: CTA rank gets [c0, c1), warp w gets [w0, w1) inside it.
    const int64_t per_cta = (S + nctas - 1) / nctas;
    const int64_t c0 = min(S, per_cta * rank);
    const int64_t c1 = min(S, c0 + per_cta);
    const int64_t per_warp = (c1 - c0 + kMetaWarps - 1) / kMetaWarps;
    const int64_t w0 = min(c1, c0 + per_warp * warp);
    const int64_t w1 = min(c1, w0 + per_warp);
    int *my_cnt = wcnt + warp * E;

    for (int i = tid; i < kMetaWarps * E; i += kMetaThreads) wcnt[i] = 0;
    if (tid == 0) sm.bad = 0;
    __syncthreads();

    pdl_wait_prior_grids();

    // ---- phase 1: per-warp histograms of the warp's slots
    for (int64_t base = w0; base < w1; base += 32) {
        const int64_t s = base + lane;
        int e = -1;
        if (s < w1) {
            e = topk_idx[s];
            if (e < 0 || e >= E) {
                sm.bad = 1;
                e = -1;
            }
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my_cnt[e] += __popc(peers);
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
        int e = -1;
        if (s < w1) {
            e = topk_idx[s];
            if (e < 0 || e >= E) e = -1;
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        const uint32_t below = peers & ((1u << lane) - 1u);
        if (s < w1) {
            if (e >= 0) {
                const int r = my_cnt[e] + __popc(below);
                row_map[s] = r;
                if (src_slot) src_slot[r] = static_cast<int32_t>(s);
            } else {
                row_map[s] = -1;
            }
        }
        __syncwarp();
        if (e >= 0 && below == 0) my_cnt[e] += __popc(peers);
        __syncwarp();
    }

    if (sm.bad && tid == 0) report_status(status, MOE_ERR_BAD_INDEX);
    pdl_launch_dependents();
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

template <bool kBf16Out, bool kFp8>
__global__ void __launch_bounds__(kPermWarps * 32) permute_kernel(
    const uint4 *__restrict__ X, const int32_t *__restrict__ row_map, int64_t N, int H, int K,
    uint4 *__restrict__ Xp, uint8_t *__restrict__ Xq, float *__restrict__ Xs, int32_t *status)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunks = H >> 3;          // 16-byte chunks per row
    const int64_t rows = N * K;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kPermWarps;

    pdl_wait_prior_grids();

    bool bad = false;
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * kPermWarps + warp; n < N; n += nwarps) {
        int my_row = -1;
        if (lane < K) {
            my_row = row_map[n * K + lane];
            if (my_row < 0 || my_row >= rows) {
                bad = true;
                my_row = -1;
            }
        }
        const uint4 *src = X + n * chunks;
        for (int c0 = 0; c0 < chunks; c0 += 64) {
            // two independent 16-byte loads per lane in flight
            const int ca = c0 + lane, cb = c0 + 32 + lane;
            const bool va = ca < chunks, vb = cb < chunks;
            uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
            if (va) xa = __ldcs(src + ca);
            if (vb) xb = __ldcs(src + cb);

            uint2 qa = make_uint2(0, 0), qb = qa;
            float sa = 0.f, sb = 0.f;
            if constexpr (kFp8) {
                // lanes 0-15 and 16-31 each hold one 128-element block
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint4 x = half ? xb : xa;
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
                    // power-of-two scale: t = fl32(max(amax, 1e-4) * fl32(1/448)),
                    // s = t's exponent, bumped when t has a non-zero mantissa
                    const float t = __fmul_rn(fmaxf(amax, 1e-4f), __uint_as_float(kRcp448Bits));
                    const uint32_t tb = __float_as_uint(t);
                    const uint32_t sbits = (tb & 0x7F800000u) + ((tb & 0x007FFFFFu) ? 0x00800000u : 0u);
                    const float s = __uint_as_float(sbits);
                    const float inv_s = __uint_as_float((254u - (sbits >> 23)) << 23);  // exact 1/s
                    uint2 q;
                    q.x = f32x2_to_e4m3x2(f[0] * inv_s, f[1] * inv_s) |
                          (f32x2_to_e4m3x2(f[2] * inv_s, f[3] * inv_s) << 16);
                    q.y = f32x2_to_e4m3x2(f[4] * inv_s, f[5] * inv_s) |
                          (f32x2_to_e4m3x2(f[6] * inv_s, f[7] * inv_s) << 16);
                    if (half) {
                        qb = q;
                        sb = s;
                    } else {
                        qa = q;
                        sa = s;
                    }
                }
            }
            for (int k = 0; k < K; ++k) {
                const int r = __shfl_sync(0xffffffffu, my_row, k);
                if (r < 0) continue;
                if constexpr (kBf16Out) {
                    uint4 *dst = Xp + static_cast<int64_t>(r) * chunks;
                    if (va) __stcs(dst + ca, xa);
                    if (vb) __stcs(dst + cb, xb);
                }
                if constexpr (kFp8) {
                    uint2 *qdst = reinterpret_cast<uint2 *>(Xq + static_cast<int64_t>(r) * H);
                    if (va) __stcs(qdst + ca, qa);
                    if (vb) __stcs(qdst + cb, qb);
                    const int nb = H >> 7;
                    if ((lane & 15) == 0) {
                        if (va) Xs[static_cast<int64_t>(r) * nb + (ca >> 4)] = sa;
                        if (vb) Xs[static_cast<int64_t>(r) * nb + (cb >> 4)] = sb;
                    }
                }
            }
        }
    }
    if (bad) report_status(status, MOE_ERR_BAD_INDEX);
    pdl_launch_dependents();
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
    const int64_t S = N * K;
    const size_t smem = sizeof(MetaSmem) + sizeof(int) * kMetaWarps * E;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    const int cl = meta_cluster_size(S);
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
    return cudaLaunchKernelEx(&cfg, dispatch_meta_kernel, topk_idx, S, E, counts, offsets, row_map, src_slot,
                              status);
}

cudaError_t launch_permute(const void *X, const int32_t *row_map, int64_t N, int H, int K, void *X_perm,
                           void *X_fp8, float *X_scale, int32_t *status, cudaStream_t stream)
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
    if (X_perm && X_fp8)
        return cudaLaunchKernelEx(&cfg, permute_kernel<true, true>, x, row_map, N, H, K, xp, xq, X_scale, status);
    if (X_fp8)
        return cudaLaunchKernelEx(&cfg, permute_kernel<false, true>, x, row_map, N, H, K, xp, xq, X_scale, status);
    return cudaLaunchKernelEx(&cfg, permute_kernel<true, false>, x, row_map, N, H, K, xp, xq, X_scale, status);
}

}  // namespace moe
