/*
 * The library used from plain C (no Python, no torch): route -> dispatch -> combine through the
 * C ABI of include/moe_route.h, then route + dispatch as one call, on device buffers from
 * cudaMalloc.  The checks need no oracle:
 *   - every token has K distinct experts in [0, E), and its renormalised weights sum to 1;
 *   - sum(expert_counts) == N*K, expert_offsets is their exclusive scan, and row_map is a
 *     permutation of [0, N*K) that sends every slot into its expert's range;
 *   - every permuted row is the bit pattern of its token's row of X;
 *   - with the expert outputs Y = X_perm, the combine gives sum_k w_k * X[n] = X[n] (to bf16
 *     rounding), because the weights sum to 1;
 *   - moe_route_dispatch gives the same ids, weights and dispatch as the two calls;
 *   - moe_combine_residual with residual = X gives 2 X (to bf16 rounding);
 *   - moe_route_stats gives the same ids and weights, the dispatch's expert counts,
 *     and each token's logsumexp (checked against one taken here in fp64);
 *   - moe_load_stats gives the mean, max/mean, P95/mean and z-loss of those
 *     counts and logsumexps as defined.
 * Prints "ok" and returns 0, or prints the first failure and returns 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "moe_route.h"

#define N_TOK 1000
#define HID 512
#define NEXP 32
#define TOPK 2

static int fail(const char *what)
{
    printf("FAIL: %s\n", what);
    return 1;
}

#define CUDA_OK(x)                                                      \
    do {                                                                \
        if ((x) != cudaSuccess) return fail(#x);                        \
    } while (0)
#define MOE_OK_(x)                                                      \
    do {                                                                \
        moe_status st_ = (x);                                           \
        if (st_ != MOE_OK) {                                            \
            printf("%s: %s\n", #x, moe_status_string(st_));             \
            return 1;                                                   \
        }                                                               \
    } while (0)

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite) */
static uint16_t to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* uniform in (-1, 1) from a 64-bit LCG */
static uint64_t lcg = 0x9E3779B97F4A7C15ull;
static float uniform(void)
{
    lcg = lcg * 6364136223846793005ull + 1442695040888963407ull;
    return (float)((double)(lcg >> 11) / 9007199254740992.0) * 2.0f - 1.0f;
}

int main(void)
{
    const int64_t N = N_TOK;
    const int H = HID, E = NEXP, K = TOPK;
    const int64_t S = N * K;
    uint16_t *hX = malloc(sizeof(uint16_t) * N * H), *hW = malloc(sizeof(uint16_t) * H * E);
    for (int64_t i = 0; i < N * H; ++i) hX[i] = to_bf16(uniform() * 1.7f);
    for (int64_t i = 0; i < (int64_t)H * E; ++i) hW[i] = to_bf16(uniform() * 1.7f / sqrtf((float)H));

    void *X, *W, *Xp, *Xp2, *out, *ws;
    int32_t *idx, *idx2, *cnt, *cnt2, *off, *off2, *rmap, *rmap2, *src, *src2, *status;
    float *w, *w2;
    const size_t wsb = moe_dispatch_workspace_size(N, E, K);
    CUDA_OK(cudaMalloc(&X, sizeof(uint16_t) * N * H));
    CUDA_OK(cudaMalloc(&W, sizeof(uint16_t) * H * E));
    CUDA_OK(cudaMalloc(&Xp, sizeof(uint16_t) * S * H));
    CUDA_OK(cudaMalloc(&Xp2, sizeof(uint16_t) * S * H));
    CUDA_OK(cudaMalloc(&out, sizeof(uint16_t) * N * H));
    CUDA_OK(cudaMalloc(&ws, wsb));
    CUDA_OK(cudaMalloc((void **)&idx, 4 * S));
    CUDA_OK(cudaMalloc((void **)&idx2, 4 * S));
    CUDA_OK(cudaMalloc((void **)&w, 4 * S));
    CUDA_OK(cudaMalloc((void **)&w2, 4 * S));
    CUDA_OK(cudaMalloc((void **)&cnt, 4 * E));
    CUDA_OK(cudaMalloc((void **)&cnt2, 4 * E));
    CUDA_OK(cudaMalloc((void **)&off, 4 * (E + 1)));
    CUDA_OK(cudaMalloc((void **)&off2, 4 * (E + 1)));
    CUDA_OK(cudaMalloc((void **)&rmap, 4 * S));
    CUDA_OK(cudaMalloc((void **)&rmap2, 4 * S));
    CUDA_OK(cudaMalloc((void **)&src, 4 * S));
    CUDA_OK(cudaMalloc((void **)&src2, 4 * S));
    CUDA_OK(cudaMalloc((void **)&status, 4));
    CUDA_OK(cudaMemcpy(X, hX, sizeof(uint16_t) * N * H, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(W, hW, sizeof(uint16_t) * H * E, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemset(ws, 0, wsb));
    CUDA_OK(cudaMemset(status, 0, 4));

    cudaStream_t s;
    CUDA_OK(cudaStreamCreate(&s));
    moe_stream_t ms = (moe_stream_t)s;
    MOE_OK_(moe_route(X, W, NULL, N, H, E, K, 1, idx, w, status, ms));
    MOE_OK_(moe_dispatch(idx, X, N, H, E, K, cnt, off, rmap, src, Xp, NULL, NULL, status, ws, wsb, ms));
    /* expert outputs Y = the permuted rows themselves */
    MOE_OK_(moe_combine(Xp, rmap, w, N, H, K, out, status, ms));
    int launches = 0;
    MOE_OK_(moe_route_dispatch(X, W, NULL, N, H, E, K, 1, idx2, w2, cnt2, off2, rmap2, src2, Xp2, status, ws, wsb,
                               &launches, ms));
    CUDA_OK(cudaStreamSynchronize(s));

    int32_t st;
    CUDA_OK(cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost));
    if (st != 0) return fail(moe_status_string((moe_status)st));

    int32_t *hi = malloc(4 * S), *hi2 = malloc(4 * S), *hc = malloc(4 * E), *ho = malloc(4 * (E + 1));
    int32_t *hr = malloc(4 * S), *hr2 = malloc(4 * S), *hs = malloc(4 * S), *hs2 = malloc(4 * S);
    int32_t *hc2 = malloc(4 * E), *ho2 = malloc(4 * (E + 1));
    float *hw = malloc(4 * S), *hw2 = malloc(4 * S);
    uint16_t *hp = malloc(sizeof(uint16_t) * S * H), *hp2 = malloc(sizeof(uint16_t) * S * H);
    uint16_t *hout = malloc(sizeof(uint16_t) * N * H);
    CUDA_OK(cudaMemcpy(hi, idx, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hi2, idx2, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hw, w, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hw2, w2, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hc, cnt, 4 * E, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hc2, cnt2, 4 * E, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(ho, off, 4 * (E + 1), cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(ho2, off2, 4 * (E + 1), cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hr, rmap, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hr2, rmap2, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hs, src, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hs2, src2, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hp, Xp, sizeof(uint16_t) * S * H, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hp2, Xp2, sizeof(uint16_t) * S * H, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hout, out, sizeof(uint16_t) * N * H, cudaMemcpyDeviceToHost));

    /* route: K distinct experts per token, weights summing to 1 */
    for (int64_t n = 0; n < N; ++n) {
        double sum = 0.0;
        for (int k = 0; k < K; ++k) {
            const int e = hi[n * K + k];
            if (e < 0 || e >= E) return fail("expert id out of range");
            for (int j = 0; j < k; ++j)
                if (hi[n * K + j] == e) return fail("repeated expert");
            sum += hw[n * K + k];
        }
        if (fabs(sum - 1.0) > 1e-5) return fail("weights do not sum to 1");
    }
    /* dispatch: counts, offsets, a permutation into the right ranges */
    int64_t total = 0;
    for (int e = 0; e < E; ++e) {
        if (ho[e] != total) return fail("offsets are not the exclusive scan of the counts");
        total += hc[e];
    }
    if (total != S || ho[E] != S) return fail("sum(counts) != N*K");
    char *seen = calloc((size_t)S, 1);
    for (int64_t q = 0; q < S; ++q) {
        const int32_t r = hr[q];
        const int e = hi[q];
        if (r < 0 || r >= S || seen[r]) return fail("row_map is not a permutation");
        seen[r] = 1;
        if (r < ho[e] || r >= ho[e + 1]) return fail("a slot outside its expert's rows");
        if (hs[r] != q) return fail("src_slot is not the inverse of row_map");
        if (memcmp(hp + (int64_t)r * H, hX + (q / K) * H, sizeof(uint16_t) * H) != 0)
            return fail("a permuted row differs from its token's row");
    }
    /* combine with Y = X_perm: out[n] = X[n] to bf16 rounding */
    for (int64_t i = 0; i < N * H; ++i) {
        const float x = from_bf16(hX[i]), o = from_bf16(hout[i]);
        if (fabsf(o - x) > 1e-2f * fabsf(x) + 1e-6f) return fail("combine differs from X");
    }
    /* route + dispatch as one call: the same results */
    if (memcmp(hi, hi2, 4 * S) != 0 || memcmp(hw, hw2, 4 * S) != 0) return fail("moe_route_dispatch routes differently");
    if (memcmp(hc, hc2, 4 * E) != 0 || memcmp(ho, ho2, 4 * (E + 1)) != 0 || memcmp(hr, hr2, 4 * S) != 0 ||
        memcmp(hs, hs2, 4 * S) != 0 || memcmp(hp, hp2, sizeof(uint16_t) * S * H) != 0)
        return fail("moe_route_dispatch dispatches differently");

    /* combine with the residual connection, residual = X: out = X + X */
    void *out2;
    CUDA_OK(cudaMalloc(&out2, sizeof(uint16_t) * N * H));
    MOE_OK_(moe_combine_residual(Xp, rmap, w, X, N, H, K, out2, status, ms));
    /* router statistics (renorm on), then the load statistics of its counts */
    int32_t *idx3, *cnt3;
    float *w3, *lse, *stats;
    CUDA_OK(cudaMalloc((void **)&idx3, 4 * S));
    CUDA_OK(cudaMalloc((void **)&w3, 4 * S));
    CUDA_OK(cudaMalloc((void **)&cnt3, 4 * E));
    CUDA_OK(cudaMalloc((void **)&lse, 4 * N));
    CUDA_OK(cudaMalloc((void **)&stats, 4 * 4));
    const float z_coef = 1e-3f;
    MOE_OK_(moe_route_stats(X, W, NULL, N, H, E, K, 1, idx3, w3, lse, cnt3, status, MOE_ROUTE_AUTO, ms));
    MOE_OK_(moe_load_stats(cnt3, E, lse, N, z_coef, stats, ms));
    CUDA_OK(cudaStreamSynchronize(s));
    CUDA_OK(cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost));
    if (st != 0) return fail(moe_status_string((moe_status)st));

    uint16_t *hout2 = malloc(sizeof(uint16_t) * N * H);
    int32_t *hi3 = malloc(4 * S), *hc3 = malloc(4 * E);
    float *hw3 = malloc(4 * S), *hl = malloc(4 * N), hst[4];
    CUDA_OK(cudaMemcpy(hout2, out2, sizeof(uint16_t) * N * H, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hi3, idx3, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hw3, w3, 4 * S, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hc3, cnt3, 4 * E, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hl, lse, 4 * N, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hst, stats, sizeof(hst), cudaMemcpyDeviceToHost));

    for (int64_t i = 0; i < N * H; ++i) {
        const float x2 = 2.0f * from_bf16(hX[i]), o = from_bf16(hout2[i]);
        if (fabsf(o - x2) > 1e-2f * fabsf(x2) + 1e-6f) return fail("combine with residual differs from 2 X");
    }
    if (memcmp(hi, hi3, 4 * S) != 0 || memcmp(hw, hw3, 4 * S) != 0) return fail("moe_route_stats routes differently");
    if (memcmp(hc, hc3, 4 * E) != 0) return fail("router histogram differs from the dispatch counts");
    /* logsumexp of the logits, taken here in fp64 from the same bf16 operands */
    for (int64_t n = 0; n < N; ++n) {
        double L[NEXP], m = -INFINITY, z = 0.0;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h) acc += (double)from_bf16(hX[n * H + h]) * (double)from_bf16(hW[h * E + e]);
            L[e] = acc;
            if (acc > m) m = acc;
        }
        for (int e = 0; e < E; ++e) z += exp(L[e] - m);
        const double ref = m + log(z);
        if (fabs((double)hl[n] - ref) > 1e-3 + 1e-5 * fabs(ref)) return fail("logsumexp differs from fp64");
    }
    /* load statistics: the mean, max/mean, P95/mean (linear interpolation) and z-loss */
    double mean = (double)S / E, cmax = 0.0, zsum = 0.0;
    int32_t sorted[NEXP];
    memcpy(sorted, hc3, sizeof(sorted));
    for (int i = 1; i < E; ++i)   /* insertion sort of E counts */
        for (int j = i; j > 0 && sorted[j - 1] > sorted[j]; --j) {
            const int32_t t = sorted[j];
            sorted[j] = sorted[j - 1];
            sorted[j - 1] = t;
        }
    cmax = sorted[E - 1];
    const double pos = 0.95 * (E - 1);
    const int lo = (int)pos;
    const double p95 = sorted[lo] + (pos - lo) * ((lo + 1 < E ? sorted[lo + 1] : sorted[lo]) - sorted[lo]);
    for (int64_t n = 0; n < N; ++n) zsum += (double)hl[n] * (double)hl[n];
    const double zloss = (double)z_coef * zsum / (double)N;
    if (fabs(hst[3] - mean) > 1e-6 * mean) return fail("load stats: mean");
    if (fabs(hst[0] - cmax / mean) > 1e-6 * (cmax / mean)) return fail("load stats: max / mean");
    if (fabs(hst[1] - p95 / mean) > 1e-6 * (p95 / mean)) return fail("load stats: P95 / mean");
    if (fabs(hst[2] - zloss) > 1e-5 * zloss + 1e-9) return fail("load stats: z-loss");

    printf("ok (moe_route_dispatch: %d launch%s)\n", launches, launches == 1 ? "" : "es");
    return 0;
}
