// route_simt.cu -- CUDA-core router: one warp per token.
//
// Used for shapes the tensor-core router does not take (E % 8 != 0, where
// the gate weight rows are not 16-byte multiples and cannot be TMA-tiled) and
// as an independent second implementation in the tests.
//
// Method (moe-engine page, "moe-engine：面向万卡集群的稀疏MoE训练基础设施",
// section 融合Triton路由内核): logits = tokens @ gate_w, softmax over the E
// experts, K rounds of selection, renormalisation of the K weights.  Here the
// E logits of a token are spread over the 32 lanes of a warp (lane l owns
// experts l, l+32, ...), and each selection round is a warp-wide argmax by
// shuffles, ties to the lower expert index.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kSimtWarps = 8;
constexpr int kMaxE = 256;
constexpr int kPerLane = kMaxE / 32;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// (v, i) ranks above (bv, bi): larger value, or equal value and lower index.
__device__ __forceinline__ bool ranks_above(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kSimtWarps * 32) route_simt_kernel(
    const uint16_t *__restrict__ X, const uint16_t *__restrict__ W, const float *__restrict__ bias, int64_t N,
    int H, int E, int K, int renorm, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
    float *__restrict__ lse, int32_t *__restrict__ counts)
{
    __shared__ float logits_s[kSimtWarps][kMaxE];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    float *L = logits_s[warp];
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kSimtWarps;

    pdl_wait_prior_grids();

    for (int64_t n = static_cast<int64_t>(blockIdx.x) * kSimtWarps + warp; n < N; n += nwarps) {
        const uint4 *xrow = reinterpret_cast<const uint4 *>(X + n * H);
        const int nchunks = H >> 3;  // 8 bf16 per 16-byte chunk
        // ---- logits, 32 experts at a time: lane-partial sums, then warp sums
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int ne = min(32, E - e0);
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.f;
            for (int c = lane; c < nchunks; c += 32) {
                const uint4 xv = __ldg(xrow + c);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    const float x = (p & 1) ? bf16_hi(xw[p >> 1]) : bf16_lo(xw[p >> 1]);
                    const uint16_t *wrow = W + static_cast<int64_t>(c * 8 + p) * E + e0;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < ne) acc[j] = fmaf(x, __uint_as_float(static_cast<uint32_t>(__ldg(wrow + j)) << 16), acc[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                float s = acc[j];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == j && j < ne) {
                    float v = s + (bias ? bias[e0 + j] : 0.f);
                    L[e0 + j] = isnan(v) ? -INFINITY : v;
                }
            }
        }
        __syncwarp();
        // ---- K rounds of warp-wide argmax
        float mine[kPerLane];
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            mine[i] = e < E ? L[e] : -INFINITY;
        }
        uint32_t taken = 0;  // bit i: expert lane + 32 i already chosen
        float sel_v = -INFINITY, first_v = -INFINITY, sum_sel = 0.f;
        int sel_i = -1;
        float my_v = 0.f;
        int my_i = -1;
        for (int k = 0; k < K; ++k) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && ranks_above(mine[i], e, bv, bi)) {
                    bv = mine[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ranks_above(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (k == 0) first_v = bv;
            sel_v = bv;
            sel_i = bi;
            const float p = expf(sel_v - first_v);
            sum_sel += p;
            if (lane == k) {
                my_v = p;
                my_i = sel_i;
            }
        }
        float denom = sum_sel;
        if (!renorm || lse) {
            // the full softmax denominator: sum over all experts of exp(logit - max)
            float z = 0.f;
#pragma unroll
            for (int i = 0; i < kPerLane; ++i)
                if (lane + 32 * i < E && mine[i] != -INFINITY) z += expf(mine[i] - first_v);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            if (!renorm) denom = z;
            if (lse && lane == 0) lse[n] = first_v == -INFINITY ? -INFINITY : first_v + logf(z);
        }
        if (lane < K) {
            topk_idx[n * K + lane] = my_i;
            topk_w[n * K + lane] = my_v / denom;
            if (counts && my_i >= 0 && my_i < E) atomicAdd(counts + my_i, 1);
        }
        __syncwarp();
    }
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_route_simt(const RouteArgs &a, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int sms = device_sm_count(dev);
    const int64_t blocks_needed = (a.N + kSimtWarps - 1) / kSimtWarps;
    const int grid = static_cast<int>(blocks_needed < int64_t(sms) * 8 ? blocks_needed : int64_t(sms) * 8);
    route_simt_kernel<<<grid, kSimtWarps * 32, 0, stream>>>(
        static_cast<const uint16_t *>(a.X), static_cast<const uint16_t *>(a.W), a.bias, a.N, a.H, a.E, a.K,
        a.renorm, a.topk_idx, a.topk_w, a.lse, a.counts);
    return cudaGetLastError();
}

}  // namespace moe
