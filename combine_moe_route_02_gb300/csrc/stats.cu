// stats.cu -- expert-load statistics of the router (moe-engine page,
// "moe-engine：面向万卡集群的稀疏MoE训练基础设施", section 专家负载均衡): the
// imbalance ratio max/mean of the per-expert slot counts, the 95th percentile
// of the counts over the mean, and a z-loss of weight z_coef over the per-token
// logsumexp of the logits (the page regularises with weight 1e-3).
//
// One CTA: the E <= 256 counts are sorted in shared memory (bitonic network)
// for the percentile, and the squares of the N logsumexp values are summed in
// fp64 in a fixed order (per-thread strided sums, then a fixed tree), so the
// result does not depend on scheduling.  This runs once per step next to the
// router, off the bandwidth-bound path.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kStatThreads = 256;  // also the sort width (E <= 256)

__global__ void __launch_bounds__(kStatThreads) load_stats_kernel(const int32_t *__restrict__ counts, int E,
                                                                  const float *__restrict__ lse, int64_t N,
                                                                  float z_coef, float *__restrict__ stats)
{
    __shared__ int key[kStatThreads];
    __shared__ double part[kStatThreads / 32];
    __shared__ long long tot[kStatThreads / 32];
    __shared__ int mx[kStatThreads / 32];
    const int t = threadIdx.x;
    const int warp = t >> 5;
    const int lane = t & 31;

    pdl_wait_prior_grids();

    const int c = t < E ? counts[t] : 0;
    key[t] = t < E ? c : 0x7fffffff;  // padding sorts to the end
    long long s = c;
    int m = c;
    double z = 0.0;
    if (lse != nullptr)
        for (int64_t i = t; i < N; i += kStatThreads) {
            const double v = lse[i];
            z += v * v;
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        z += __shfl_xor_sync(0xffffffffu, z, o);
    }
    if (lane == 0) {
        tot[warp] = s;
        mx[warp] = m;
        part[warp] = z;
    }
    // ascending bitonic sort of the padded counts
    for (int size = 2; size <= kStatThreads; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            const int l = t ^ stride;
            if (l > t) {
                const int a = key[t], b = key[l];
                const bool up = (t & size) == 0;
                if ((a > b) == up) {
                    key[t] = b;
                    key[l] = a;
                }
            }
        }
    }
    __syncthreads();
    if (t == 0) {
        long long total = 0;
        int mxc = 0;
        double zs = 0.0;
        for (int w = 0; w < kStatThreads / 32; ++w) {
            total += tot[w];
            mxc = max(mxc, mx[w]);
            zs += part[w];
        }
        const double mean = static_cast<double>(total) / E;
        const double pos = 0.95 * (E - 1);
        const int lo = static_cast<int>(floor(pos));
        const int hi = lo + 1 < E ? lo + 1 : E - 1;
        const double p95 = key[lo] + (pos - lo) * static_cast<double>(key[hi] - key[lo]);
        stats[0] = mean > 0.0 ? static_cast<float>(mxc / mean) : 0.f;
        stats[1] = mean > 0.0 ? static_cast<float>(p95 / mean) : 0.f;
        stats[2] = (lse != nullptr && N > 0) ? static_cast<float>(static_cast<double>(z_coef) * zs / N) : 0.f;
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
