// combine.cu -- weighted gather of the K expert rows of every token back to
// token order (forward_aggregate, PithTrain page
// "一万行Python构建MoE训练栈：解构4D并行、DualPipeV调度与FP8算子",
// §6.1 模型协议先行):  out[n,:] = sum_k w[n,k] * Y[row_map[n*K+k], :], and,
// with the residual connection of the same method, + residual[n,:].
//
// One warp per token, 16-byte vectors: every lane gathers the same 16-byte
// column chunk from the K rows (independent loads, all in flight together,
// with the residual chunk), accumulates in fp32 in k order, adds the residual,
// rounds to bf16 (nearest even) and stores.  A lane reads its residual chunk
// before it writes the same chunk of out, so out may be the residual buffer
// itself (an in-place update of the residual stream).
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

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 &r)
{
    const uint32_t v[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        acc[2 * p] += __uint_as_float(v[p] << 16);
        acc[2 * p + 1] += __uint_as_float(v[p] & 0xFFFF0000u);
    }
}

// The output rows: streamed through L2 (evict-first), or, where the whole
// output fits in L2 next to what is still in use (`keep`), stored with the
// default write-back policy for the kernel that reads them next.
__device__ __forceinline__ void st_out(uint4 *p, const uint4 &v, int keep)
{
    if (keep)
        *p = v;
    else
        __stcs(p, v);
}

// KT > 0: K known at compile time -- every lane issues the loads of CPL
// chunks x KT rows before the first FMA (CPL * KT <= 16 uint4 in flight per
// lane).  KT == 0: runtime K, one chunk at a time.  RES: add residual[n,:]
// after the weighted sum (out and residual may be the same buffer, so
// neither is declared restrict).
template <int KT, int CPL, bool RES>
__global__ void __launch_bounds__(kCombWarps * 32) combine_kernel(
    const uint4 *__restrict__ Y, const int32_t *__restrict__ row_map, const float *__restrict__ w, int64_t N,
    int H, int K_rt, const uint4 *residual, uint4 *out, int32_t *status, int keep)
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
        const uint4 *res = RES ? residual + n * chunks : nullptr;
        if constexpr (KT > 0) {
            const uint4 *yr[KT];
            float wk[KT];
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                yr[k] = Y + static_cast<int64_t>(__shfl_sync(0xffffffffu, my_row, k)) * chunks;
                wk[k] = __shfl_sync(0xffffffffu, my_w, k);
            }
            for (int base = 0; base < chunks; base += 32 * CPL) {
                uint4 y[CPL][KT];
                uint4 rr[RES ? CPL : 1];
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const int c = base + lane + 32 * j;
#pragma unroll
                    for (int k = 0; k < KT; ++k) y[j][k] = c < chunks ? __ldcs(yr[k] + c) : make_uint4(0, 0, 0, 0);
                    if constexpr (RES) rr[j] = c < chunks ? __ldcs(res + c) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const int c = base + lane + 32 * j;
                    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < KT; ++k) fma_bf16x8(acc, y[j][k], wk[k]);
                    if constexpr (RES) add_bf16x8(acc, rr[j]);
                    if (c < chunks) st_out(dst + c, pack_bf16x8(acc), keep);
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
                if constexpr (RES) {
                    if (v) add_bf16x8(acc, __ldcs(res + c));
                }
                if (v) st_out(dst + c, pack_bf16x8(acc), keep);
            }
        }
    }
    if (bad) report_status(status, MOE_ERR_BAD_INDEX);
    pdl_launch_dependents();
}

int pow2_chunks_per_lane(int chunks, int cap)
{
    int c = 1;
    while (c < cap && 32 * c < chunks) c <<= 1;
    return c;
}

}  // namespace

template <bool RES>
cudaError_t launch_combine_t(const void *Y, const int32_t *row_map, const float *w, const void *residual,
                             int64_t N, int H, int K, void *out, int32_t *status, cudaStream_t stream)
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
    const uint4 *res = static_cast<const uint4 *>(residual);
    uint4 *o = static_cast<uint4 *>(out);
    const int chunks = H / 8;
    const int keep = keep_in_l2(N * 2 * static_cast<int64_t>(H), dev) ? 1 : 0;
#define MOE_COMBINE_LAUNCH(KK, C)                                                              \
    if ((err = prefer_l1_carveout<combine_kernel<KK, C, RES>>(dev)) != cudaSuccess) return err; \
    return cudaLaunchKernelEx(&cfg, combine_kernel<KK, C, RES>, y, row_map, w, N, H, K, res, o, status, keep)
    switch (K) {
    case 1:
        switch (pow2_chunks_per_lane(chunks, 16)) {
        case 1: MOE_COMBINE_LAUNCH(1, 1);
        case 2: MOE_COMBINE_LAUNCH(1, 2);
        case 4: MOE_COMBINE_LAUNCH(1, 4);
        case 8: MOE_COMBINE_LAUNCH(1, 8);
        default: MOE_COMBINE_LAUNCH(1, 16);
        }
    case 2:
        switch (pow2_chunks_per_lane(chunks, 8)) {
        case 1: MOE_COMBINE_LAUNCH(2, 1);
        case 2: MOE_COMBINE_LAUNCH(2, 2);
        case 4: MOE_COMBINE_LAUNCH(2, 4);
        default: MOE_COMBINE_LAUNCH(2, 8);
        }
    case 4:
        switch (pow2_chunks_per_lane(chunks, 4)) {
        case 1: MOE_COMBINE_LAUNCH(4, 1);
        case 2: MOE_COMBINE_LAUNCH(4, 2);
        default: MOE_COMBINE_LAUNCH(4, 4);
        }
    case 8:
        switch (pow2_chunks_per_lane(chunks, 2)) {
        case 1: MOE_COMBINE_LAUNCH(8, 1);
        default: MOE_COMBINE_LAUNCH(8, 2);
        }
    default: MOE_COMBINE_LAUNCH(0, 1);
    }
#undef MOE_COMBINE_LAUNCH
}

cudaError_t launch_combine(const void *Y, const int32_t *row_map, const float *w, const void *residual, int64_t N,
                           int H, int K, void *out, int32_t *status, cudaStream_t stream)
{
    if (residual) return launch_combine_t<true>(Y, row_map, w, residual, N, H, K, out, status, stream);
    return launch_combine_t<false>(Y, row_map, w, nullptr, N, H, K, out, status, stream);
}

}  // namespace moe
