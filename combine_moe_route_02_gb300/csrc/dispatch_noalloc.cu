// dispatch_noalloc.cu -- moe_dispatch_noalloc: the one-launch dispatch with its
// scratch memory built into the library instead of passed in by the caller.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they dispatch tokens -- an engine that plans all of its device memory up front
// and forbids allocation afterwards, code running in a host callback or in a
// context where cudaMalloc would block or implicitly synchronise the device,
// or a C caller with no allocator of its own to hand a workspace from.  They
// still pass the input and output buffers; only the scratch comes from here.
//
// The scratch is one file-scope device array of kScratchBytes (a 256-byte
// grid-barrier header plus one int32 count per (CTA, expert) for up to 1024
// CTAs and 256 experts, i.e. 1 MiB + 256 bytes).  Every GPU that loads the
// library holds it until the process exits.  Host code cannot use the array's
// name as a device address: the first call on each device resolves the address
// with cudaGetSymbolAddress (with that device current) and caches it.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr size_t kScratchBytes = 256 + 1024ull * 256ull * sizeof(int32_t);

static __device__ __align__(256) unsigned char g_dispatch_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_dispatch_scratch on `device` (the current device),
// resolved once per device; nullptr if the lookup failed.
void *scratch_address(int device)
{
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    static bool done[kMaxDevices] = {};
    if (device < 0 || device >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[device]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;  // not cached: a later call retries
        }
        addr[device] = p;
        done[device] = true;
    }
    return addr[device];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status moe_dispatch_noalloc(const int32_t *topk_idx, const void *X, int64_t N, int H, int E,
                                                   int K, int32_t *expert_counts, int32_t *expert_offsets,
                                                   int32_t *row_map, int32_t *src_slot, void *X_perm, void *X_fp8,
                                                   float *X_scale, int32_t *status_word, moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_dispatch_noalloc");
    // Every argument check of moe_dispatch runs first, on the host: a rejected
    // call makes no CUDA call and queues nothing on the stream.
    const moe_status st = dispatch_check(topk_idx, X, N, H, E, K, expert_counts, expert_offsets, row_map, src_slot,
                                         X_perm, X_fp8, X_scale, MOE_SCALE_FP32, status_word, nullptr, 0);
    if (st != MOE_OK) return st;
    if (N == 0)   // zero counts and offsets; no scratch needed
        return moe_dispatch(topk_idx, X, N, H, E, K, expert_counts, expert_offsets, row_map, src_slot, X_perm, X_fp8,
                            X_scale, status_word, nullptr, 0, stream);
    int dev = 0;
    if (const cudaError_t ge = cudaGetDevice(&dev); ge != cudaSuccess) return from_cuda(ge);
    // Sizes beyond what the built-in scratch serves: one launch takes
    // min(N, SMs) CTAs and at most 16384 slots per CTA, i.e.
    // ceil(N / min(N, SMs)) * K <= 16384.
    const int64_t sms = device_sm_count(dev);
    const int64_t ctas = N < sms ? N : sms;
    const int64_t tok_per = (N + ctas - 1) / ctas;
    if (tok_per * K > 16384 || ctas > 1024 || 256 + static_cast<size_t>(ctas) * E * sizeof(int32_t) > kScratchBytes)
        return MOE_ERR_UNSUPPORTED;
    void *scratch = scratch_address(dev);
    if (!scratch) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the grid-barrier counters
    // must start at zero, the per-CTA counts are overwritten before use.
    if (const cudaError_t me = cudaMemsetAsync(scratch, 0, 256, s); me != cudaSuccess) return from_cuda(me);
    return moe_dispatch(topk_idx, X, N, H, E, K, expert_counts, expert_offsets, row_map, src_slot, X_perm, X_fp8,
                        X_scale, status_word, scratch, kScratchBytes, s);
}
