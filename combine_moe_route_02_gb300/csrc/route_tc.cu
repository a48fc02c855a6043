// route_tc.cu -- the fused router on the 5th-generation tensor cores.
//
// Method (moe-engine page, "moe-engine：面向万卡集群的稀疏MoE训练基础设施",
// section 融合Triton路由内核): logits = tokens @ gate_w, softmax over E,
// top-K, renorm -- in one pass over X, so the logits never reach HBM.
//
// GB300 design (not the page's 64x64 SRAM tiling):
//   * one CTA per 128-token tile, 6 warps:
//       warp 0    TMA producer: X tile [128 x 64] and gate-weight slab
//                 [64 x EP] per K-step, 128-byte swizzle, into a ring of
//                 `stages` shared-memory slots (mbarrier full/empty pairs);
//       warp 1    MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16 -> fp32),
//                 M = 128, N = E rounded up to 16, four K = 16 steps per
//                 slot; the fp32 logits accumulate in TMEM (128 lanes x N
//                 columns) and never leave the SM;
//       warps 2-5 epilogue: each thread owns one token (TMEM lane), reads its
//                 E logits with tcgen05.ld, adds the bias, keeps the running
//                 top-K in registers (one pass, K compare-exchange steps per
//                 candidate -- the same K largest, in the same order and with
//                 the same tie rule as K rounds of selection), then forms the
//                 weights with an fp32 softmax.
//   * X is K-major (row-major [N,H]); the gate weight [H,E] is read as it is
//     stored, as an MN-major B operand (E contiguous), so no transpose pass.
//   * Every mbarrier wait is bounded (2 s of %globaltimer); on expiry the CTA
//     records MOE_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM, exits.
#include <math.h>

#include <atomic>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;        // tokens per CTA (UMMA M)
constexpr int kBK = 64;         // bf16 per 128-byte swizzle row (one K-step slot)
constexpr int kThreads = 192;   // 6 warps
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KiB X tile per slot
constexpr uint32_t kBBoxBytes = kBK * 64 * 2; // 8 KiB per 64-expert gate box

struct TcSmemTail {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ bool ranks_above(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 2) route_tc_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
    const float *__restrict__ bias, int N, int H, int E, int K, int renorm, int EP, int NP, int stages,
    uint32_t tmem_cols, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w, int32_t *status)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t b_slot_bytes = static_cast<uint32_t>(EP) * kBK * 2;
    unsigned char *a_base = smem;
    unsigned char *b_base = smem + static_cast<size_t>(stages) * kABytes;
    TcSmemTail &tail =
        *reinterpret_cast<TcSmemTail *>(b_base + static_cast<size_t>(stages) * b_slot_bytes);
    float *bias_s = reinterpret_cast<float *>(&tail + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kBM;
    const int nk = (H + kBK - 1) / kBK;
    volatile int *abort_flag = &tail.abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&tail.full[s], 1);
            mbar_init(&tail.empty[s], 1);
        }
        mbar_init(&tail.acc_full, 1);
        mbar_init(&tail.drain, 1);
        tail.abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(&tail.tmem_base, tmem_cols);
        tmem_relinquish();
    }
    // inputs may come from the previous kernel in the stream (programmatic launch)
    pdl_wait_prior_grids();
    for (int e = threadIdx.x; e < EP; e += kThreads) bias_s[e] = (bias != nullptr && e < E) ? bias[e] : 0.f;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = tail.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_x = l2_policy_evict_first();
            const uint64_t pol_w = l2_policy_evict_last();
            int issued = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % stages;
                const uint32_t use = static_cast<uint32_t>(kb / stages);
                if (!mbar_wait_bounded(&tail.empty[s], (use & 1u) ^ 1u, abort_flag)) break;
                mbar_arrive_expect_tx(&tail.full[s], kABytes + b_slot_bytes);
                tma_load_2d(a_base + static_cast<size_t>(s) * kABytes, &tmX, &tail.full[s], kb * kBK, m0, pol_x);
                for (int j = 0; j < EP / 64; ++j)
                    tma_load_2d(b_base + static_cast<size_t>(s) * b_slot_bytes + j * kBBoxBytes, &tmW,
                                &tail.full[s], j * 64, kb * kBK, pol_w);
                issued = kb + 1;
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA exits
                for (int kb = issued - stages < 0 ? 0 : issued - stages; kb < issued; ++kb) {
                    volatile int no_abort = 0;
                    mbar_wait_bounded(&tail.full[kb % stages], static_cast<uint32_t>(kb / stages) & 1u,
                                      &no_abort);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc_bf16_f32(kBM, static_cast<uint32_t>(NP), 0u, 1u);
            const uint32_t a0 = smem_u32(a_base);
            const uint32_t b0 = smem_u32(b_base);
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % stages;
                const uint32_t use = static_cast<uint32_t>(kb / stages);
                if (!mbar_wait_bounded(&tail.full[s], use & 1u, abort_flag)) break;
                tc_fence_after_sync();
                const uint32_t a_s = a0 + static_cast<uint32_t>(s) * kABytes;
                const uint32_t b_s = b0 + static_cast<uint32_t>(s) * b_slot_bytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    // A: K-major, 128-byte rows, 8-row groups 1024 B apart; +32 B per K=16 step
                    const uint64_t a_desc = make_smem_desc_sw128(a_s + kk * 32, 16, 1024);
                    // B: MN-major, 64-expert atoms 8 KiB apart (LBO), 8-row K groups 1024 B
                    // apart (SBO); +16 rows x 128 B per K=16 step
                    const uint64_t b_desc = make_smem_desc_sw128(b_s + kk * 2048, kBBoxBytes, 1024);
                    tc_mma_f16(tmem_base, a_desc, b_desc, idesc, (kb | kk) != 0 ? 1u : 0u);
                }
                tc_commit(&tail.empty[s]);  // slot free once these MMAs have read it
            }
            tc_commit(&tail.acc_full);      // logits complete
            tc_commit(&tail.drain);
            volatile int no_abort = 0;
            mbar_wait_bounded(&tail.drain, 0, &no_abort);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int n = m0 + q * 32 + lane;
        if (mbar_wait_bounded(&tail.acc_full, 0, abort_flag)) {
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            float bv[KMAX];
            int bi[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                bv[j] = -INFINITY;
                bi[j] = 0x7fffffff;
            }
            for (int c0 = 0; c0 < NP; c0 += 32) {
                float v[32];
                tmem_ld_32x32b_x32(taddr + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int e = c0 + j;
                    if (e >= E) break;
                    float x = v[j] + bias_s[e];
                    if (isnan(x)) x = -INFINITY;
                    if (ranks_above(x, e, bv[KMAX - 1], bi[KMAX - 1])) {
                        float cv = x;
                        int ci = e;
#pragma unroll
                        for (int t = 0; t < KMAX; ++t) {
                            const bool up = ranks_above(cv, ci, bv[t], bi[t]);
                            const float ov = bv[t];
                            const int oi = bi[t];
                            bv[t] = up ? cv : ov;
                            bi[t] = up ? ci : oi;
                            cv = up ? ov : cv;
                            ci = up ? oi : ci;
                        }
                    }
                }
            }
            const float m = bv[0];
            float denom = 0.f;
            if (renorm) {
#pragma unroll
                for (int t = 0; t < KMAX; ++t)
                    if (t < K) denom += expf(bv[t] - m);
            } else {
                for (int c0 = 0; c0 < NP; c0 += 32) {
                    float v[32];
                    tmem_ld_32x32b_x32(taddr + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = c0 + j;
                        if (e >= E) break;
                        const float x = v[j] + bias_s[e];
                        if (!isnan(x)) denom += expf(x - m);
                    }
                }
            }
            if (n < N) {
#pragma unroll
                for (int t = 0; t < KMAX; ++t) {
                    if (t < K) {
                        topk_idx[static_cast<int64_t>(n) * K + t] = bi[t];
                        topk_w[static_cast<int64_t>(n) * K + t] = expf(bv[t] - m) / denom;
                    }
                }
            }
        }
        tc_fence_before_sync();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
    if (threadIdx.x == 0 && tail.abort) report_status(status, MOE_ERR_TIMEOUT);
    pdl_launch_dependents();
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
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
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

struct TcPlan {
    int EP, NP, stages;
    uint32_t tmem_cols;
    size_t smem;
};

TcPlan plan_for(int E)
{
    TcPlan p;
    p.EP = (E + 63) / 64 * 64;
    p.NP = (E + 15) / 16 * 16;
    const uint32_t slot = kABytes + static_cast<uint32_t>(p.EP) * kBK * 2;
    // two CTAs per SM while that still leaves >= 2 slots (~100 KiB each)
    int st = static_cast<int>((100u * 1024u) / slot);
    if (st > 8) st = 8;
    if (st < 2) st = 2;
    p.stages = st;
    uint32_t cols = 32;
    while (cols < static_cast<uint32_t>(p.NP)) cols <<= 1;
    p.tmem_cols = cols;
    p.smem = 1024 + static_cast<size_t>(st) * slot + sizeof(TcSmemTail) + sizeof(float) * p.EP;
    return p;
}

template <int KMAX>
cudaError_t launch_tc_k(const RouteArgs &a, const TcPlan &p, const CUtensorMap &tmX, const CUtensorMap &tmW,
                        cudaStream_t stream, int dev)
{
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = 1ull << (dev & 63);
    cudaError_t err;
    if (!(configured.load() & bit)) {
        err = cudaFuncSetAttribute(route_tc_kernel<KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   227 * 1024);
        if (err != cudaSuccess) return err;
        configured.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>((a.N + kBM - 1) / kBM), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_tc_kernel<KMAX>, tmX, tmW, a.bias, static_cast<int>(a.N), a.H, a.E, a.K,
                              a.renorm, p.EP, p.NP, p.stages, p.tmem_cols, a.topk_idx, a.topk_w, a.status);
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

cudaError_t launch_route_tc(const RouteArgs &a, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const TcPlan p = plan_for(a.E);
    CUtensorMap tmX, tmW;
    if (!encode_2d_bf16(&tmX, a.X, static_cast<uint64_t>(a.H), static_cast<uint64_t>(a.N), kBK, kBM))
        return cudaErrorInvalidValue;
    if (!encode_2d_bf16(&tmW, a.W, static_cast<uint64_t>(a.E), static_cast<uint64_t>(a.H), 64, kBK))
        return cudaErrorInvalidValue;
    if (a.K <= 2) return launch_tc_k<2>(a, p, tmX, tmW, stream, dev);
    if (a.K <= 4) return launch_tc_k<4>(a, p, tmX, tmW, stream, dev);
    if (a.K <= 8) return launch_tc_k<8>(a, p, tmX, tmW, stream, dev);
    return launch_tc_k<16>(a, p, tmX, tmW, stream, dev);
}

}  // namespace moe
