// dispatch_ep.cu -- expert-parallel dispatch metadata with token deduplication,
// for the tokens of one GPU (PithTrain page, "一万行Python构建MoE训练栈：解构4D并行、
// DualPipeV调度与FP8算子", §8.2 O(n) counting sort 替代 O(n log n) argsort:
// fused_dedup_prepare_dispatch counts tokens per expert and per EP rank, builds
// the prefix sums and the send metadata, and does the dedup scatter, the
// counting sort and expand_idx).  The all-to-all that would move the rows is
// outside this library.
//
// Experts are split over R = ep_size ranks, P = E / R consecutive experts each.
// A token goes to a rank once however many of its experts live there.  Three
// launches on the caller's stream:
//   1. the one-launch counting-sort dispatch with the experts as keys
//      (metadata only): expert counts/offsets, row_map, and the inverse map
//      (kept in expand_idx for step 3);
//   2. the same kernel with the EP ranks as keys, where a slot whose rank
//      already appeared earlier in its token is ignored: rank counts/offsets,
//      the send row of every first-occurrence slot (in slot_send_row), the
//      first slot of every send row (kept in send_token for step 3), and the
//      dedup'd send rows X_send[row] = X[token];
//   3. a fix-up kernel: every other slot takes the send row of the first slot
//      of its token with the same rank, send_token becomes token ids,
//      expand_idx maps each expert-ordered slot to its token's index inside
//      its rank's block of send rows, and send_meta is filled.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kFixThreads = 256;

__global__ void __launch_bounds__(kFixThreads) ep_fixup_kernel(
    const int32_t *__restrict__ topk_idx, int64_t N, int E, int K, int P, int R,
    const int32_t *__restrict__ expert_counts, const int32_t *__restrict__ expert_offsets,
    const int32_t *__restrict__ rank_counts, const int32_t *__restrict__ rank_offsets, int32_t *slot_send_row,
    int32_t *send_token, int32_t *expand_idx, int32_t *__restrict__ send_meta)
{
    pdl_wait_prior_grids();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kFixThreads;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kFixThreads + threadIdx.x;
    const int64_t slots = N * K;

    // the send row of a slot = the row its token's first slot with the same rank
    // received (first-occurrence entries are final and are not written here)
    for (int64_t s = t0; s < slots; s += stride) {
        if (slot_send_row[s] >= 0) continue;
        const int e = topk_idx[s];
        if (e < 0 || e >= E) continue;
        const int64_t base = s - s % K;
        for (int64_t j = base; j < s; ++j) {
            const int ej = topk_idx[j];
            if (ej >= 0 && ej < E && ej / P == e / P) {
                slot_send_row[s] = slot_send_row[j];
                break;
            }
        }
    }
    // send rows: first slot -> token
    const int64_t rows = rank_offsets[R];
    for (int64_t q = t0; q < rows; q += stride) send_token[q] = send_token[q] / K;
    // expert-ordered slots: index of the token in its rank's received rows
    const int64_t erows = expert_offsets[E];
    for (int64_t q = t0; q < erows; q += stride) {
        const int64_t s = expand_idx[q];  // the slot of row q (inverse map of the expert pass)
        const int e = topk_idx[s];
        const int r = e / P;
        int64_t j = s - s % K;
        while (j < s) {  // the token's first slot on rank r holds the send row
            const int ej = topk_idx[j];
            if (ej >= 0 && ej < E && ej / P == r) break;
            ++j;
        }
        expand_idx[q] = slot_send_row[j] - rank_offsets[r];
    }
    for (int64_t i = t0; i < static_cast<int64_t>(R) * (P + 1); i += stride) {
        const int r = static_cast<int>(i / (P + 1));
        const int j = static_cast<int>(i % (P + 1));
        send_meta[i] = j == 0 ? rank_counts[r] : expert_counts[r * P + j - 1];
    }
    pdl_launch_dependents();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status moe_dispatch_ep(const int32_t *topk_idx, const void *X, int64_t N, int H, int E, int K,
                                              int ep_size, int32_t *expert_counts, int32_t *expert_offsets,
                                              int32_t *row_map, int32_t *rank_counts, int32_t *rank_offsets,
                                              int32_t *send_token, int32_t *slot_send_row, int32_t *expand_idx,
                                              int32_t *send_meta, void *X_send, int32_t *status_word,
                                              void *workspace, size_t workspace_bytes, moe_stream_t stream)
{
    NvtxRange nvtx_range("moe_dispatch_ep");
    if (E < 1 || E > 256 || K < 1 || K > 16 || K > E || N < 0) return MOE_ERR_INVALID_ARG;
    if (N > 0 && N > (static_cast<int64_t>(0x7fffffff) - 1) / K) return MOE_ERR_INVALID_ARG;
    if (ep_size < 1 || ep_size > E || E % ep_size != 0) return MOE_ERR_INVALID_ARG;
    if (!expert_counts || !expert_offsets || !rank_counts || !rank_offsets || !send_meta) return MOE_ERR_INVALID_ARG;
    if (N > 0 && (!topk_idx || !row_map || !send_token || !slot_send_row || !expand_idx))
        return MOE_ERR_INVALID_ARG;
    if (X_send && !X) return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < fused_workspace_bytes(E)) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MOE_ERR_MISALIGNED;
    const void *ptrs4[] = {topk_idx, expert_counts, expert_offsets, row_map, rank_counts, rank_offsets,
                           send_token, slot_send_row, expand_idx, send_meta, status_word};
    for (const void *q : ptrs4)
        if (reinterpret_cast<uintptr_t>(q) & 3u) return MOE_ERR_MISALIGNED;
    if (X) {
        if (!X_send || H < 1) return MOE_ERR_INVALID_ARG;
        if (H % 8 != 0 || (reinterpret_cast<uintptr_t>(X) & 15u) || (reinterpret_cast<uintptr_t>(X_send) & 15u))
            return MOE_ERR_MISALIGNED;
    }
    const int R = ep_size;
    const int P = E / R;
    int dev = 0;
    if (const cudaError_t ge = cudaGetDevice(&dev); ge != cudaSuccess) return from_cuda(ge);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) {
        cudaError_t me = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s);
        if (me == cudaSuccess) me = cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), s);
        if (me == cudaSuccess) me = cudaMemsetAsync(rank_counts, 0, sizeof(int32_t) * R, s);
        if (me == cudaSuccess) me = cudaMemsetAsync(rank_offsets, 0, sizeof(int32_t) * (R + 1), s);
        if (me == cudaSuccess) me = cudaMemsetAsync(send_meta, 0, sizeof(int32_t) * R * (P + 1), s);
        return from_cuda(me);
    }
    if (!dispatch_fused_supported(N, K, dev)) return MOE_ERR_UNSUPPORTED;
    // 1. experts as keys, metadata only; the inverse map goes to expand_idx
    cudaError_t e = launch_dispatch_fused(topk_idx, nullptr, N, 0, E, K, expert_counts, expert_offsets, row_map,
                                          expand_idx, nullptr, nullptr, nullptr, 0, status_word, workspace,
                                          workspace_bytes, s, 0);
    if (e != cudaSuccess) return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED : from_cuda(e);
    // 2. EP ranks as keys with deduplication; the first slot of each send row goes to send_token.
    // A large send-row copy runs as its own permute launch (more warps storing), before the
    // fix-up fills in the slots that take no row of their own
    const int64_t max_rows = N * (K < R ? K : R);
    const bool copy_apart = X != nullptr && N * 2 * static_cast<int64_t>(H) + max_rows * 2 * H >= kPermuteApartBytes;
    e = launch_dispatch_fused(topk_idx, copy_apart ? nullptr : X, N, X ? H : 0, R, K, rank_counts, rank_offsets,
                              slot_send_row, send_token, X_send, nullptr, nullptr, 0, status_word, workspace,
                              workspace_bytes, s, P);
    if (e != cudaSuccess) return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED : from_cuda(e);
    if (copy_apart) {
        e = launch_permute(X, slot_send_row, N, H, K, X_send, nullptr, nullptr, 0, status_word, s, true);
        if (e != cudaSuccess) return from_cuda(e);
    }
    // 3. fix-up
    const int sms = device_sm_count(dev);
    const int64_t need = (N * K + kFixThreads - 1) / kFixThreads;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(need < 2 * sms ? (need < 1 ? 1 : need) : 2 * sms), 1, 1);
    cfg.blockDim = dim3(kFixThreads, 1, 1);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, ep_fixup_kernel, topk_idx, N, E, K, P, R, static_cast<const int32_t *>(expert_counts),
                           static_cast<const int32_t *>(expert_offsets), static_cast<const int32_t *>(rank_counts),
                           static_cast<const int32_t *>(rank_offsets), slot_send_row, send_token, expand_idx,
                           send_meta);
    return from_cuda(e);
}
