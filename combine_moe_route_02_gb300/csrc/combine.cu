// combine.cu -- weighted gather of the K expert rows of every token back to
// token order (the weighted part of forward_aggregate, PithTrain page
// "一万行Python构建MoE训练栈：解构4D并行、DualPipeV调度与FP8算子",
// §6.1 模型协议先行):  out[n,:] = sum_k w[n,k] * Y[row_map[n*K+k], :].
//
// One warp per token, 16-byte vectors: every lane gathers the same 16-byte
// column chunk from the K rows (independent loads, all in flight together),
// accumulates in fp32 in k order, rounds to bf16 (nearest even) and stores.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kCombWarps = 8;

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], const uint4 &y, float w)
{
    const uint32_t v[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        acc[2 * p] = fmaf(w, __uint_as_float(v[p] << 16), acc[2 * p]);
        acc[2 * p + 1] = fmaf(w, __uint_as_float(v[p] & 0xFFFF0000u), acc[2 * p + 1]);
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8])
{
    uint4 o;
    uint32_t *po = &o.x;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * p], acc[2 * p + 1]);
        po[p] = *reinterpret_cast<const uint32_t *>(&b);
    }
    return o;
}

// KT > 0: K known at compile time (loads of all K rows unrolled); KT == 0: runtime K.
template <int KT>
__global__ void __launch_bounds__(kCombWarps * 32) combine_kernel(
    const uint4 *__restrict__ Y, const int32_t *__restrict__ row_map, const float *__restrict__ w, int64_t N,
    int H, int K_rt, uint4 *__restrict__ out, int32_t *status)
{
    const int K = KT > 0 ? KT : K_rt;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunks = H >> 3;
    const int64_t rows = N * K;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kCombWarps;

    pdl_wait_prior_grids();

    bool bad = false;
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * kCombWarps + warp; n < N; n += nwarps) {
        int my_row = 0;
        float my_w = 0.f;
        if (lane < K) {
            my_row = row_map[n * K + lane];
            my_w = w[n * K + lane];
            if (my_row < 0 || my_row >= rows) {
                bad = true;
                my_row = 0;
                my_w = 0.f;
            }
        }
        uint4 *dst = out + n * chunks;
        if constexpr (KT > 0) {
            int r[KT];
            float wk[KT];
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                r[k] = __shfl_sync(0xffffffffu, my_row, k);
                wk[k] = __shfl_sync(0xffffffffu, my_w, k);
            }
            constexpr int U = KT <= 2 ? 4 : (KT <= 4 ? 2 : 1);
            for (int c0 = lane; c0 < chunks; c0 += 32 * U) {
                uint4 y[U][KT];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int k = 0; k < KT; ++k) {
                        const int c = c0 + 32 * u;
                        y[u][k] = c < chunks ? __ldcs(Y + static_cast<int64_t>(r[k]) * chunks + c)
                                             : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + 32 * u;
                    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < KT; ++k) fma_bf16x8(acc, y[u][k], wk[k]);
                    if (c < chunks) __stcs(dst + c, pack_bf16x8(acc));
                }
            }
        } else {
            for (int c0 = 0; c0 < chunks; c0 += 32) {  // warp-uniform trip count
                const int c = c0 + lane;
                const bool v = c < chunks;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int k = 0; k < K; ++k) {
                    const int r = __shfl_sync(0xffffffffu, my_row, k);
                    const float wk = __shfl_sync(0xffffffffu, my_w, k);
                    if (v) fma_bf16x8(acc, __ldcs(Y + static_cast<int64_t>(r) * chunks + c), wk);
                }
                if (v) __stcs(dst + c, pack_bf16x8(acc));
            }
        }
    }
    if (bad) report_status(status, MOE_ERR_BAD_INDEX);
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_combine(const void *Y, const int32_t *row_map, const float *w, int64_t N, int H, int K,
                           void *out, int32_t *status, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int sms = device_sm_count(dev);
    const int64_t need = (N + kCombWarps - 1) / kCombWarps;
    const int64_t cap = int64_t(sms) * 8;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(need < cap ? need : cap), 1, 1);
    cfg.blockDim = dim3(kCombWarps * 32, 1, 1);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint4 *y = static_cast<const uint4 *>(Y);
    uint4 *o = static_cast<uint4 *>(out);
    switch (K) {
    case 1: return cudaLaunchKernelEx(&cfg, combine_kernel<1>, y, row_map, w, N, H, K, o, status);
    case 2: return cudaLaunchKernelEx(&cfg, combine_kernel<2>, y, row_map, w, N, H, K, o, status);
    case 4: return cudaLaunchKernelEx(&cfg, combine_kernel<4>, y, row_map, w, N, H, K, o, status);
    case 8: return cudaLaunchKernelEx(&cfg, combine_kernel<8>, y, row_map, w, N, H, K, o, status);
    default: return cudaLaunchKernelEx(&cfg, combine_kernel<0>, y, row_map, w, N, H, K, o, status);
    }
}

}  // namespace moe
