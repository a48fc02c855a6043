// moe_internal.cuh -- shared device helpers and launcher declarations of the
// GB300 (sm_103a) MoE routing library.  Inline PTX for mbarriers, TMA and the
// 5th-generation tensor cores (tcgen05 + TMEM).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe_route.h"

namespace moe {

// ---------------------------------------------------------------------------
// Device error word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report_status(int32_t *status_word, int32_t code)
{
    if (status_word) atomicCAS(status_word, 0, code);
}

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Lanes of the warp whose key equals this lane's key, for keys in [0, 512):
// one ballot per key bit, all independent (cheaper here than __match_any_sync).
__device__ __forceinline__ uint32_t same_key_lanes(int key)
{
    uint32_t m = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 9; ++b) {
        const bool bit = (key >> b) & 1;
        const uint32_t bal = __ballot_sync(0xffffffffu, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
}

// Grid-barrier counters in global memory (acquire load, release add).
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_add_release_gpu(unsigned *p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete.  Gives up (returns false) when
// *abort becomes non-zero or after kWaitLimitNs, in which case it raises
// *abort itself so that every other role of the CTA stops too.  sleep_ns > 0
// parks the thread between polls (for waits that are not latency critical,
// so that pollers leave issue slots to the producer and MMA warps).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                  uint32_t sleep_ns = 0)
{
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (sleep_ns) __nanosleep(sleep_ns);
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                            int32_t c1, uint64_t cache_policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(cache_policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                            int32_t c1, int32_t c2, uint64_t cache_policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(cache_policy)
        : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Plain bulk copy shared -> global (16-byte aligned addresses, size a multiple
// of 16), tracked in this thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(gdst)),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

// Wait until every bulk copy this thread committed has completed (its reads of
// shared memory and its writes to global memory).
__device__ __forceinline__ void bulk_commit_and_wait_all()
{
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group 0;" ::: "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads
// ---------------------------------------------------------------------------
// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at `dst`.  Whole-warp instruction.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 inputs, fp32 acc).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (base lane + t), columns [col, col+32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 4 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x4(uint32_t taddr, float (&v)[4])
{
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier over `count` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (sm_100 family format):
// start address, leading/stride byte offsets (all >> 4), version 1 at bit 46,
// base offset 0, swizzle mode in bits 61..63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t make_smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation and bf16 A/B.
// a_mn_major / b_mn_major select MN-major (transposed) operand layouts.
__host__ __device__ constexpr uint32_t make_idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t a_mn_major,
                                                           uint32_t b_mn_major)
{
    return (1u << 4)                 // D format: f32
           | (1u << 7)               // A format: bf16
           | (1u << 10)              // B format: bf16
           | (a_mn_major << 15)      // A major
           | (b_mn_major << 16)      // B major
           | ((N >> 3) << 17)        // N / 8
           | ((M >> 4) << 24);       // M / 16
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait_prior_grids()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Launchers (host side), one per kernel family.  They assume validated
// arguments and return the launch's cudaError_t.
// ---------------------------------------------------------------------------
struct RouteArgs {
    const void *X;
    const void *W;
    const float *bias;
    int64_t N;
    int H, E, K, renorm;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *status;
    float *lse = nullptr;        // [N] per-token logsumexp of the logits, or nullptr
    int32_t *counts = nullptr;   // [E] selections per expert, accumulated (zeroed first), or nullptr
};

// Outputs of the dispatch part of a route + dispatch launch.
struct FuseArgs {
    int32_t *counts, *offsets, *row_map, *src_slot;
    void *X_perm;      // bf16 rows in expert order, or nullptr (metadata only)
    void *workspace;   // fused_workspace_bytes(E) bytes, 256-byte aligned, barrier counters zero
};

// Whether the tensor-core router can take this shape on the current device.
bool route_tc_supported(const RouteArgs &a, int device);
// Route and dispatch in one cooperative launch (split-mode router, every CTA
// resident).  cudaErrorNotSupported when this shape or device cannot take it;
// nothing has been launched then.
cudaError_t launch_route_dispatch_tc(const RouteArgs &a, const FuseArgs &f, cudaStream_t stream);
cudaError_t launch_route_tc(const RouteArgs &a, cudaStream_t stream);
cudaError_t launch_route_simt(const RouteArgs &a, cudaStream_t stream);

// Expert-load statistics (one CTA): stats[0..3] = max/mean, p95/mean, z-loss, mean.
cudaError_t launch_load_stats(const int32_t *counts, int E, const float *lse, int64_t N, float z_coef,
                              float *stats, cudaStream_t stream);

cudaError_t launch_dispatch_meta(const int32_t *topk_idx, int64_t N, int E, int K, int32_t *counts,
                                 int32_t *offsets, int32_t *row_map, int32_t *src_slot, int32_t *status,
                                 cudaStream_t stream);

// Counting sort + permute in one cooperative launch; cudaErrorNotSupported when
// the problem or the workspace does not fit (the caller then falls back to the
// cluster metadata kernel + launch_permute).
cudaError_t launch_dispatch_fused(const int32_t *topk_idx, const void *X, int64_t N, int H, int E, int K,
                                  int32_t *counts, int32_t *offsets, int32_t *row_map, int32_t *src_slot,
                                  void *X_perm, void *X_fp8, void *X_scale, int scale_ue8m0, int32_t *status,
                                  void *workspace, size_t workspace_bytes, cudaStream_t stream, int ep_P = 0);
// Whether launch_dispatch_fused takes N tokens of K slots on this device.
bool dispatch_fused_supported(int64_t N, int K, int device);
size_t fused_workspace_bytes(int E);

// X_scale: fp32 [N*K, H/128], or (scale_ue8m0 != 0) one UE8M0 byte per block.
// skip_unset: a row_map entry of -1 means "no row" and is not reported.
cudaError_t launch_permute(const void *X, const int32_t *row_map, int64_t N, int H, int K, void *X_perm,
                           void *X_fp8, void *X_scale, int scale_ue8m0, int32_t *status, cudaStream_t stream,
                           bool skip_unset = false);
// Row copies at least this large run as their own launch of the permute kernel.
constexpr int64_t kPermuteApartBytes = int64_t(256) << 20;

// residual: NULL for the plain weighted combine.
cudaError_t launch_combine(const void *Y, const int32_t *row_map, const float *w, const void *residual, int64_t N,
                           int H, int K, void *out, int32_t *status, cudaStream_t stream);

// Names one C-ABI call on a profiler's timeline (NVTX push/pop; without a
// profiler attached the calls return at once).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// The status of a CUDA runtime call for the C ABI.  A failure is reported by the
// status alone: the runtime's last-error slot is cleared so that a caller's
// later, unrelated check does not see it again.
inline moe_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return MOE_OK;
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
}

// Host checks of moe_dispatch_ex's arguments (moe_api.cu); no CUDA call.  A
// NULL workspace with workspace_bytes == 0 is valid (the path without workspace).
moe_status dispatch_check(const int32_t *topk_idx, const void *X, int64_t N, int H, int E, int K,
                          const int32_t *expert_counts, const int32_t *expert_offsets, const int32_t *row_map,
                          const int32_t *src_slot, const void *X_perm, const void *X_fp8, const void *X_scale,
                          int scale_format, const int32_t *status_word, const void *workspace,
                          size_t workspace_bytes);

// Number of SMs of the current device (cached per device).
int device_sm_count(int device);
int device_cc_major(int device);
// L2 size of a device in bytes (cached per device; 1 where the attribute is missing).
int64_t device_l2_bytes(int device);
// Whether a kernel's output of `bytes` is left in L2 for the kernel that reads it
// next (default write-back stores, or the TMA's evict-normal policy for an input
// that a later kernel reads again) rather than streamed through it (evict-first):
// at most 5/8 of the L2.
bool keep_in_l2(int64_t bytes, int device);

// Ask for the L1-heavy shared-memory carve-out for a copy kernel (set once per
// device and kernel).  The row copies and the combine keep many 16-byte loads in
// flight per SM and use little shared memory; with the carve-out of a kernel that
// held most of shared memory before them (the persistent router) they ran ~15%
// slower.  A CTA placed on an SM that was never idle in between keeps that SM's
// carve-out, which is what happened when a CUDA graph replayed the step with the
// router's early launch trigger (65536 x 4096 tokens: 644 against 586 us).
template <auto *Kernel>
cudaError_t prefer_l1_carveout(int device)
{
    static std::atomic<uint64_t> done{0};
    const uint64_t bit = 1ull << (device & 63);
    if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    const cudaError_t err =
        cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxL1);
    if (err == cudaSuccess) done.fetch_or(bit, std::memory_order_relaxed);
    return err;
}

}  // namespace moe
