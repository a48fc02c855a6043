// moe_api.cu -- the C ABI of the routing library: argument validation on the
// host (before any CUDA call, so that a rejected call touches no device
// state), implementation choice, and the launches.
#include <atomic>
#include <climits>

#include "moe_internal.cuh"

namespace moe {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_cc_major[kMaxDevices];
std::atomic<int64_t> g_l2_bytes[kMaxDevices];

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

moe_status check_topk(int E, int K)
{
    if (E < 1 || E > 256) return MOE_ERR_INVALID_ARG;
    if (K < 1 || K > 16 || K > E) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// Bytes the row permute moves: X read once, K bf16 rows and/or K E4M3 rows + scales written.
int64_t permute_bytes(int64_t N, int H, int K, bool bf16, bool fp8)
{
    int64_t per_token = 2 * static_cast<int64_t>(H);
    if (bf16) per_token += 2 * static_cast<int64_t>(K) * H;
    if (fp8) per_token += static_cast<int64_t>(K) * (H + H / 32);
    return N * per_token;
}

moe_status check_rows(int64_t N, int K)
{
    if (N < 0) return MOE_ERR_INVALID_ARG;
    if (N > 0 && N > (static_cast<int64_t>(INT_MAX) - 1) / K) return MOE_ERR_INVALID_ARG;  // N*K < 2^31
    return MOE_OK;
}
}  // namespace

int device_sm_count(int device)
{
    const int d = device & (kMaxDevices - 1);
    int v = g_sm_count[d].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0) v = 1;
        g_sm_count[d].store(v, std::memory_order_relaxed);
    }
    return v;
}

int64_t device_l2_bytes(int device)
{
    const int d = device & (kMaxDevices - 1);
    int64_t v = g_l2_bytes[d].load(std::memory_order_relaxed);
    if (v <= 0) {
        int b = 0;
        if (cudaDeviceGetAttribute(&b, cudaDevAttrL2CacheSize, device) != cudaSuccess || b < 0) b = 0;
        v = b > 0 ? b : 1;
        g_l2_bytes[d].store(v, std::memory_order_relaxed);
    }
    return v;
}

bool keep_in_l2(int64_t bytes, int device)
{
    // a little over half of the cache: what the next kernel reads back stays
    // there next to the inputs still in use
    return bytes <= device_l2_bytes(device) / 8 * 5;
}

int device_cc_major(int device)
{
    const int d = device & (kMaxDevices - 1);
    int v = g_cc_major[d].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess || v <= 0)
            v = -1;
        g_cc_major[d].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(moe_status s)
{
    switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: a required pointer is NULL or a size is out of range";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: the requested implementation cannot take this shape";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: pointers must be 16-byte aligned and H a multiple of 8";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace smaller than moe_dispatch_workspace_size()";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait ran out";
    case MOE_ERR_BAD_INDEX: return "MOE_ERR_BAD_INDEX: an expert index or row index was out of range";
    }
    return "unknown moe_status";
}

int moe_abi_version(void) { return MOE_ABI_VERSION; }

moe_status moe_route_ex(const void *X, const void *W_gate, const float *bias, int64_t N, int H, int E, int K,
                        int renorm, int32_t *topk_idx, float *topk_w, int32_t *status_word, int algo,
                        moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_route");
    moe_status st = check_topk(E, K);
    if (st != MOE_OK) return st;
    if ((st = check_rows(N, K)) != MOE_OK) return st;
    if (algo < MOE_ROUTE_AUTO || algo > MOE_ROUTE_SIMT) return MOE_ERR_INVALID_ARG;
    if (H < 1) return MOE_ERR_INVALID_ARG;
    if (N == 0) return MOE_OK;
    if (!X || !W_gate || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_MISALIGNED;
    if (!aligned16(X) || !aligned16(W_gate) || !aligned4(topk_idx) || !aligned4(topk_w) ||
        (bias && !aligned4(bias)) || (status_word && !aligned4(status_word)))
        return MOE_ERR_MISALIGNED;

    RouteArgs a{X, W_gate, bias, N, H, E, K, renorm ? 1 : 0, topk_idx, topk_w, status_word};
    int dev = 0;
    if (const cudaError_t ge = cudaGetDevice(&dev); ge != cudaSuccess) return from_cuda(ge);
    const bool tc_ok = route_tc_supported(a, dev);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (algo == MOE_ROUTE_TCGEN05 && !tc_ok) return MOE_ERR_UNSUPPORTED;
    if (algo == MOE_ROUTE_SIMT || !tc_ok) return from_cuda(launch_route_simt(a, s));
    return from_cuda(launch_route_tc(a, s));
}

moe_status moe_route_stats(const void *X, const void *W_gate, const float *bias, int64_t N, int H, int E, int K,
                           int renorm, int32_t *topk_idx, float *topk_w, float *lse, int32_t *expert_counts,
                           int32_t *status_word, int algo, moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_route_stats");
    moe_status st = check_topk(E, K);
    if (st != MOE_OK) return st;
    if ((st = check_rows(N, K)) != MOE_OK) return st;
    if (algo < MOE_ROUTE_AUTO || algo > MOE_ROUTE_SIMT) return MOE_ERR_INVALID_ARG;
    if (H < 1) return MOE_ERR_INVALID_ARG;
    if ((lse && !aligned4(lse)) || (expert_counts && !aligned4(expert_counts))) return MOE_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) {
        return expert_counts ? from_cuda(cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s)) : MOE_OK;
    }
    if (!X || !W_gate || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_MISALIGNED;
    if (!aligned16(X) || !aligned16(W_gate) || !aligned4(topk_idx) || !aligned4(topk_w) ||
        (bias && !aligned4(bias)) || (status_word && !aligned4(status_word)))
        return MOE_ERR_MISALIGNED;

    RouteArgs a{X, W_gate, bias, N, H, E, K, renorm ? 1 : 0, topk_idx, topk_w, status_word};
    a.lse = lse;
    a.counts = expert_counts;
    int dev = 0;
    if (const cudaError_t ge = cudaGetDevice(&dev); ge != cudaSuccess) return from_cuda(ge);
    const bool tc_ok = route_tc_supported(a, dev);
    if (algo == MOE_ROUTE_TCGEN05 && !tc_ok) return MOE_ERR_UNSUPPORTED;
    // the kernels add their selections to the counts
    if (expert_counts) {
        const moe_status ms = from_cuda(cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s));
        if (ms != MOE_OK) return ms;
    }
    if (algo == MOE_ROUTE_SIMT || !tc_ok) return from_cuda(launch_route_simt(a, s));
    return from_cuda(launch_route_tc(a, s));
}

moe_status moe_load_stats(const int32_t *expert_counts, int E, const float *lse, int64_t N, float z_coef,
                          float *stats, moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_load_stats");
    if (E < 1 || E > 256 || N < 0) return MOE_ERR_INVALID_ARG;
    if (!expert_counts || !stats) return MOE_ERR_INVALID_ARG;
    if (!aligned4(expert_counts) || !aligned4(stats) || (lse && !aligned4(lse))) return MOE_ERR_MISALIGNED;
    return from_cuda(launch_load_stats(expert_counts, E, lse, N, z_coef, stats,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_route(const void *X, const void *W_gate, const float *bias, int64_t N, int H, int E, int K,
                     int renorm, int32_t *topk_idx, float *topk_w, int32_t *status_word, moe_stream_t stream)
{
    return moe_route_ex(X, W_gate, bias, N, H, E, K, renorm, topk_idx, topk_w, status_word, MOE_ROUTE_AUTO,
                        stream);
}

size_t moe_dispatch_workspace_size(int64_t N, int E, int K)
{
    (void)N;
    (void)K;
    if (E < 1 || E > 256) return 0;
    return fused_workspace_bytes(E);  // grid-barrier counters + one count per (CTA, expert)
}

static moe_status validate_permute(const void *X, const int32_t *row_map, int64_t N, int H, int K,
                                   const void *X_perm, const void *X_fp8, const void *X_scale, int scale_format)
{
    if (scale_format != MOE_SCALE_FP32 && scale_format != MOE_SCALE_UE8M0) return MOE_ERR_INVALID_ARG;
    if (!X || !row_map) return MOE_ERR_INVALID_ARG;
    if (!X_perm && !X_fp8) return MOE_ERR_INVALID_ARG;
    if ((X_fp8 == nullptr) != (X_scale == nullptr)) return MOE_ERR_INVALID_ARG;
    if (H < 1) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_MISALIGNED;
    if (X_fp8 && H % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (!aligned16(X) || (X_perm && !aligned16(X_perm)) || (X_fp8 && !aligned16(X_fp8)) ||
        (X_scale && scale_format == MOE_SCALE_FP32 && !aligned4(X_scale)) || !aligned4(row_map))
        return MOE_ERR_MISALIGNED;
    (void)N;
    (void)K;
    return MOE_OK;
}

}  // extern "C"

namespace moe {

// Host checks of moe_dispatch_ex's arguments; no CUDA call.  A NULL workspace
// with workspace_bytes == 0 is valid (the path without workspace).
moe_status dispatch_check(const int32_t *topk_idx, const void *X, int64_t N, int H, int E, int K,
                          const int32_t *expert_counts, const int32_t *expert_offsets, const int32_t *row_map,
                          const int32_t *src_slot, const void *X_perm, const void *X_fp8, const void *X_scale,
                          int scale_format, const int32_t *status_word, const void *workspace,
                          size_t workspace_bytes)
{
    moe_status st = check_topk(E, K);
    if (st != MOE_OK) return st;
    if ((st = check_rows(N, K)) != MOE_OK) return st;
    if (scale_format != MOE_SCALE_FP32 && scale_format != MOE_SCALE_UE8M0) return MOE_ERR_INVALID_ARG;
    if (!expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
    if (!aligned4(expert_counts) || !aligned4(expert_offsets) || (status_word && !aligned4(status_word)))
        return MOE_ERR_MISALIGNED;
    if (!X && (X_perm || X_fp8 || X_scale)) return MOE_ERR_INVALID_ARG;
    // no workspace at all selects the single-cluster path; otherwise it must be large enough
    const bool use_ws = workspace != nullptr || workspace_bytes != 0;
    if (use_ws && (!workspace || workspace_bytes < moe_dispatch_workspace_size(N, E, K))) return MOE_ERR_WORKSPACE;
    if (use_ws && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MOE_ERR_MISALIGNED;
    if (N > 0) {
        if (!topk_idx || !row_map) return MOE_ERR_INVALID_ARG;
        if (!aligned4(topk_idx) || !aligned4(row_map) || (src_slot && !aligned4(src_slot)))
            return MOE_ERR_MISALIGNED;
        if (X && (st = validate_permute(X, row_map, N, H, K, X_perm, X_fp8, X_scale, scale_format)) != MOE_OK)
            return st;
    }
    return MOE_OK;
}

}  // namespace moe

// moe_dispatch_ex; *launches receives the number of kernels launched.
static moe_status dispatch_impl(const int32_t *topk_idx, const void *X, int64_t N, int H, int E, int K,
                                int32_t *expert_counts, int32_t *expert_offsets, int32_t *row_map, int32_t *src_slot,
                                void *X_perm, void *X_fp8, void *X_scale, int scale_format, int32_t *status_word,
                                void *workspace, size_t workspace_bytes, cudaStream_t s, int *launches)
{
    *launches = 0;
    const moe_status st = dispatch_check(topk_idx, X, N, H, E, K, expert_counts, expert_offsets, row_map, src_slot,
                                         X_perm, X_fp8, X_scale, scale_format, status_word, workspace,
                                         workspace_bytes);
    if (st != MOE_OK) return st;
    const bool use_ws = workspace != nullptr || workspace_bytes != 0;
    const int ue8m0 = scale_format == MOE_SCALE_UE8M0;
    if (N == 0) {
        // no tokens: every count and offset is zero
        cudaError_t me = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s);
        if (me == cudaSuccess) me = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), s);
        return from_cuda(me);
    }
    if (use_ws) {
        // Large row copies run as a second launch: the permute kernel keeps up to
        // 64 warps per SM storing (the one-launch kernel has 16), which pays for
        // the extra launch once the copy moves a few hundred MB.
        const bool copy_apart = X != nullptr && permute_bytes(N, H, K, X_perm != nullptr, X_fp8 != nullptr) >=
                                                    kPermuteApartBytes;
        const cudaError_t f = launch_dispatch_fused(topk_idx, copy_apart ? nullptr : X, N, H, E, K, expert_counts,
                                                    expert_offsets, row_map, src_slot, X_perm, X_fp8, X_scale, ue8m0,
                                                    status_word, workspace, workspace_bytes, s);
        if (f == cudaSuccess) {
            *launches = 1;
            if (!copy_apart) return MOE_OK;
            *launches = 2;
            return from_cuda(launch_permute(X, row_map, N, H, K, X_perm, X_fp8, X_scale, ue8m0, status_word, s));
        }
        if (f != cudaErrorNotSupported) return from_cuda(f);
    }
    cudaError_t e = launch_dispatch_meta(topk_idx, N, E, K, expert_counts, expert_offsets, row_map, src_slot,
                                         status_word, s);
    if (e != cudaSuccess) return from_cuda(e);
    *launches = 1;
    if (X) {
        e = launch_permute(X, row_map, N, H, K, X_perm, X_fp8, X_scale, ue8m0, status_word, s);
        if (e != cudaSuccess) return from_cuda(e);
        *launches = 2;
    }
    return MOE_OK;
}

extern "C" {

moe_status moe_dispatch_ex(const int32_t *topk_idx, const void *X, int64_t N, int H, int E, int K,
                           int32_t *expert_counts, int32_t *expert_offsets, int32_t *row_map, int32_t *src_slot,
                           void *X_perm, void *X_fp8, void *X_scale, int scale_format, int32_t *status_word,
                           void *workspace, size_t workspace_bytes, moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_dispatch");
    int launches = 0;
    return dispatch_impl(topk_idx, X, N, H, E, K, expert_counts, expert_offsets, row_map, src_slot, X_perm, X_fp8,
                         X_scale, scale_format, status_word, workspace, workspace_bytes,
                         reinterpret_cast<cudaStream_t>(stream), &launches);
}

moe_status moe_route_dispatch(const void *X, const void *W_gate, const float *bias, int64_t N, int H, int E, int K,
                              int renorm, int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                              int32_t *expert_offsets, int32_t *row_map, int32_t *src_slot, void *X_perm,
                              int32_t *status_word, void *workspace, size_t workspace_bytes, int *launches,
                              moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_route_dispatch");
    if (launches) *launches = 0;
    moe_status st = check_topk(E, K);
    if (st != MOE_OK) return st;
    if ((st = check_rows(N, K)) != MOE_OK) return st;
    if (H < 1) return MOE_ERR_INVALID_ARG;
    if (!expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < moe_dispatch_workspace_size(N, E, K)) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MOE_ERR_MISALIGNED;
    if (!aligned4(expert_counts) || !aligned4(expert_offsets) || (status_word && !aligned4(status_word)))
        return MOE_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) {
        cudaError_t me = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s);
        if (me == cudaSuccess) me = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), s);
        return from_cuda(me);
    }
    if (!X || !W_gate || !topk_idx || !topk_w || !row_map) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_MISALIGNED;
    if (!aligned16(X) || !aligned16(W_gate) || !aligned4(topk_idx) || !aligned4(topk_w) || !aligned4(row_map) ||
        (bias && !aligned4(bias)) || (src_slot && !aligned4(src_slot)) || (X_perm && !aligned16(X_perm)))
        return MOE_ERR_MISALIGNED;

    RouteArgs a{X, W_gate, bias, N, H, E, K, renorm ? 1 : 0, topk_idx, topk_w, status_word};
    FuseArgs f{expert_counts, expert_offsets, row_map, src_slot, X_perm, workspace};
    const cudaError_t fe = launch_route_dispatch_tc(a, f, s);
    if (fe == cudaSuccess) {
        if (launches) *launches = 1;
        return MOE_OK;
    }
    if (fe != cudaErrorNotSupported) return from_cuda(fe);
    // apart: the router, then the dispatch of its ids
    if ((st = moe_route_ex(X, W_gate, bias, N, H, E, K, renorm, topk_idx, topk_w, status_word, MOE_ROUTE_AUTO,
                           stream)) != MOE_OK)
        return st;
    int disp = 0;
    st = dispatch_impl(topk_idx, X_perm ? X : nullptr, N, H, E, K, expert_counts, expert_offsets, row_map,
                       src_slot, X_perm, nullptr, nullptr, MOE_SCALE_FP32, status_word, workspace, workspace_bytes,
                       s, &disp);
    if (launches) *launches = 1 + disp;
    return st;
}

moe_status moe_dispatch(const int32_t *topk_idx, const void *X, int64_t N, int H, int E, int K,
                        int32_t *expert_counts, int32_t *expert_offsets, int32_t *row_map, int32_t *src_slot,
                        void *X_perm, void *X_fp8, float *X_scale, int32_t *status_word, void *workspace,
                        size_t workspace_bytes, moe_stream_t stream)
{
    return moe_dispatch_ex(topk_idx, X, N, H, E, K, expert_counts, expert_offsets, row_map, src_slot, X_perm, X_fp8,
                           X_scale, MOE_SCALE_FP32, status_word, workspace, workspace_bytes, stream);
}

moe_status moe_permute_ex(const void *X, const int32_t *row_map, int64_t N, int H, int K, void *X_perm,
                          void *X_fp8, void *X_scale, int scale_format, int32_t *status_word, moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_permute");
    if (K < 1 || K > 16) return MOE_ERR_INVALID_ARG;
    if (scale_format != MOE_SCALE_FP32 && scale_format != MOE_SCALE_UE8M0) return MOE_ERR_INVALID_ARG;
    moe_status st = check_rows(N, K);
    if (st != MOE_OK) return st;
    if (N == 0) return MOE_OK;
    if ((st = validate_permute(X, row_map, N, H, K, X_perm, X_fp8, X_scale, scale_format)) != MOE_OK) return st;
    if (status_word && !aligned4(status_word)) return MOE_ERR_MISALIGNED;
    return from_cuda(launch_permute(X, row_map, N, H, K, X_perm, X_fp8, X_scale, scale_format == MOE_SCALE_UE8M0,
                                    status_word, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_permute(const void *X, const int32_t *row_map, int64_t N, int H, int K, void *X_perm, void *X_fp8,
                       float *X_scale, int32_t *status_word, moe_stream_t stream)
{
    return moe_permute_ex(X, row_map, N, H, K, X_perm, X_fp8, X_scale, MOE_SCALE_FP32, status_word, stream);
}

static moe_status validate_combine(const void *Y, const int32_t *row_map, const float *topk_w, int64_t N, int H,
                                   int K, const void *out, const int32_t *status_word)
{
    if (K < 1 || K > 16) return MOE_ERR_INVALID_ARG;
    moe_status st = check_rows(N, K);
    if (st != MOE_OK) return st;
    if (H < 1) return MOE_ERR_INVALID_ARG;
    if (N == 0) return MOE_OK;
    if (!Y || !row_map || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_MISALIGNED;
    if (!aligned16(Y) || !aligned16(out) || !aligned4(row_map) || !aligned4(topk_w) ||
        (status_word && !aligned4(status_word)))
        return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

moe_status moe_combine(const void *Y, const int32_t *row_map, const float *topk_w, int64_t N, int H, int K,
                       void *out, int32_t *status_word, moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_combine");
    const moe_status st = validate_combine(Y, row_map, topk_w, N, H, K, out, status_word);
    if (st != MOE_OK || N == 0) return st;
    return from_cuda(launch_combine(Y, row_map, topk_w, nullptr, N, H, K, out, status_word,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_residual(const void *Y, const int32_t *row_map, const float *topk_w, const void *residual,
                                int64_t N, int H, int K, void *out, int32_t *status_word, moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_combine_residual");
    const moe_status st = validate_combine(Y, row_map, topk_w, N, H, K, out, status_word);
    if (st != MOE_OK || N == 0) return st;
    if (!residual) return MOE_ERR_INVALID_ARG;
    if (!aligned16(residual)) return MOE_ERR_MISALIGNED;
    return from_cuda(launch_combine(Y, row_map, topk_w, residual, N, H, K, out, status_word,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
