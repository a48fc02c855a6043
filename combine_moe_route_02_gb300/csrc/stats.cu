// stats.cu -- expert-load statistics of the router (moe-engine page,
// "moe-engine：面向万卡集群的稀疏MoE训练基础设施", section 专家负载均衡): the
// imbalance ratio max/mean of the per-expert slot counts, the 95th percentile
// of the counts over the mean, and a z-loss of weight z_coef over the per-token
// logsumexp of the logits (the page regularises with weight 1e-3).
//
// One CTA of 1024 threads: the squares of the N logsumexp values are summed in a
// fixed order (each thread a fixed set of elements, 16-byte loads several in
// flight, Kahan-compensated fp32; the per-thread sums added in fp64 in a fixed
// order), so the result does not depend on scheduling; the two order statistics the 95th percentile needs are
// found by ranking each of the E <= 256 counts against the others (ties by
// index) rather than by sorting.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kStatThreads = 1024;
constexpr int kStatBatch = 8;      // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kStatThreads) load_stats_kernel(const int32_t *__restrict__ counts, int E,
                                                                  const float *__restrict__ lse, int64_t N,
                                                                  float z_coef, float *__restrict__ stats)
{
    __shared__ int key[256];
    __shared__ double zpart[kStatThreads];
    __shared__ long long tpart[8];
    __shared__ int mpart[8];
    __shared__ int q_lo, q_hi;
    __shared__ double zsum_s;
    const int t = threadIdx.x;
    const int warp = t >> 5;
    const int lane = t & 31;

    pdl_wait_prior_grids();

    if (t < 256) key[t] = t < E ? counts[t] : 0;
    // sum of lse^2: each thread a fixed set of elements in a fixed order (16-byte
    // loads, kStatBatch in flight), Kahan-compensated in fp32 -- this GPU's fp64
    // rate is a small fraction of fp32 -- then the 1024 per-thread sums are added
    // in fp64 by one warp in a fixed order
    float zs = 0.f, zc = 0.f;
    auto kahan = [&](float v) {
        const float y = v * v - zc;
        const float u = zs + y;
        zc = (u - zs) - y;
        zs = u;
    };
    if (lse != nullptr) {
        int64_t done = 0;
        if ((reinterpret_cast<uintptr_t>(lse) & 15u) == 0) {
            const float4 *l4 = reinterpret_cast<const float4 *>(lse);
            const int64_t n4 = N >> 2;
            for (int64_t base = t; base < n4; base += static_cast<int64_t>(kStatThreads) * kStatBatch) {
                float4 v[kStatBatch];
#pragma unroll
                for (int u = 0; u < kStatBatch; ++u) {
                    const int64_t i = base + static_cast<int64_t>(u) * kStatThreads;
                    v[u] = i < n4 ? __ldcs(l4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kStatBatch; ++u) {
                    kahan(v[u].x);
                    kahan(v[u].y);
                    kahan(v[u].z);
                    kahan(v[u].w);
                }
            }
            done = n4 << 2;
        }
        for (int64_t i = done + t; i < N; i += kStatThreads) kahan(lse[i]);
    }
    zpart[t] = static_cast<double>(zs) - static_cast<double>(zc);
    __syncthreads();  // key[] and zpart[] ready

    // total, maximum, and the order statistics around position 0.95 (E - 1): the
    // count whose rank (ties broken by index) equals lo or hi
    const double pos = 0.95 * (E - 1);
    const int lo = static_cast<int>(floor(pos));
    const int hi = lo + 1 < E ? lo + 1 : E - 1;
    if (t < 256) {
        const int c = t < E ? key[t] : 0;
        long long sum = c;
        int mx = c;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        if (lane == 0) {
            tpart[warp] = sum;
            mpart[warp] = mx;
        }
        if (t < E) {
            int rank = 0;
            for (int j = 0; j < E; ++j) {
                const int kj = key[j];
                rank += (kj < c || (kj == c && j < t)) ? 1 : 0;
            }
            if (rank == lo) q_lo = c;
            if (rank == hi) q_hi = c;
        }
    }
    if (warp == 8) {
        double acc = 0.0;
        for (int i = lane; i < kStatThreads; i += 32) acc += zpart[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) zsum_s = acc;
    }
    __syncthreads();
    if (t == 0) {
        const double zsum = zsum_s;
        long long total = 0;
        int mxc = 0;
        for (int w = 0; w < 8; ++w) {
            total += tpart[w];
            mxc = max(mxc, mpart[w]);
        }
        const double mean = static_cast<double>(total) / E;
        const double p95 = q_lo + (pos - lo) * static_cast<double>(q_hi - q_lo);
        stats[0] = mean > 0.0 ? static_cast<float>(mxc / mean) : 0.f;
        stats[1] = mean > 0.0 ? static_cast<float>(p95 / mean) : 0.f;
        stats[2] = (lse != nullptr && N > 0) ? static_cast<float>(static_cast<double>(z_coef) * zsum / N) : 0.f;
        stats[3] = static_cast<float>(mean);
    }
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_load_stats(const int32_t *counts, int E, const float *lse, int64_t N, float z_coef, float *stats,
                              cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kStatThreads, 1, 1);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, load_stats_kernel, counts, E, lse, N, z_coef, stats);
}

}  // namespace moe
