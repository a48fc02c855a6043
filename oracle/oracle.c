/*
 * oracle.c -- plain, slow, obviously correct CPU statement of the MoE routing
 * hot path: route (logits, softmax, top-K, renorm), dispatch (stable counting
 * sort by expert), row permute with optional E4M3 1x128 block quantisation,
 * and the weighted combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check of __graft_entry__ and
 * the CPU-baseline leg of bench.py use it.  It shares no code, header, table
 * or constant with the CUDA library.
 *
 * Floating point is carried in fp64 (IEEE double) unless a step is defined by
 * the pages in fp32 (the E4M3 scale rule), in which case fp32 rounding is
 * reproduced explicitly with (float) casts of exact fp64 products.
 *
 * Sources (page title, section):
 *   [moe-engine]  "moe-engine：面向万卡集群的稀疏MoE训练基础设施" (zingnex.cn),
 *                 section 融合Triton路由内核: tokens @ gate_w -> softmax ->
 *                 top-K -> renorm; K-round selection sort;
 *                 section 专家负载均衡: imbalance max/mean, 95th percentile,
 *                 z-loss regularisation with weight 1e-3;
 *                 section 实验结果与性能数据 / Token守恒验证:
 *                 sum(dispatch_cnt) == N*K.
 *   [PithTrain]   "一万行Python构建MoE训练栈：解构4D并行、DualPipeV调度与FP8算子"
 *                 (yunpan.plus), §8.2 O(n) counting sort 替代 O(n log n) argsort
 *                 (histogram -> prefix sum -> scatter + expand_idx);
 *                 §7.2 架构感知的量化核 (_compute_fp8_scale: clamp amax at
 *                 1e-4, multiply by 1/448 in fp32, power-of-two ceiling by the
 *                 exponent-bump bit rule, or, on the e8m0 branch, rounding
 *                 toward +infinity to a UE8M0 exponent byte);
 *                 §6.1 模型协议先行 (forward_aggregate: weighted expert output
 *                 plus the residual connection).
 *   [C++ trainer] devpress.csdn.net C++/CUDA LLM trainer page, §6.2 FP8量化格式
 *                 (E4M3: 1 sign, 4 exponent, 3 mantissa bits, range +-448).
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes of the repository):
 *   - top-K is chosen on the logits (softmax is monotone), K rounds of
 *     "largest remaining", strict '>' so that ties go to the lower expert
 *     index; output slots are in descending order; NaN counts as -inf;
 *   - renorm divides each selected probability by the sum of the selected
 *     probabilities, with no epsilon;
 *   - expert_offsets has E+1 entries, offsets[E] == N*K;
 *   - row_map[slot] = row of the expert-contiguous buffer, where slot = n*K+k,
 *     rows ordered by (expert, slot) -- the stable argsort of the slots by
 *     expert; src_slot is its inverse;
 *   - the E4M3 block is 1x128 along H; the stored scale s is the dequant
 *     multiplier (x ~ q*s) and q = E4M3_rn_satfinite(x/s);
 *   - combine sums in fp64 and rounds once to bf16 (round to nearest even).
 *
 * Build: gcc -O2 -std=c11 -fopenmp -shared -fPIC oracle.c -lm
 * (OpenMP only spreads independent tokens over host threads; it changes no
 * arithmetic.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_BAD_INDEX = 7, ORACLE_NO_MEM = 8 };

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Round a double to the nearest bf16 (ties to even), straight from the
 * double value (one rounding).  bf16 keeps 8 significant bits, the binary32
 * exponent range, and subnormals with quantum 2^-133.
 */
uint16_t oracle_f64_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    if (isinf(x))
        return x > 0 ? 0x7F80 : 0xFF80;
    if (x == 0.0)
        return signbit(x) ? 0x8000 : 0x0000;
    int ex;
    frexp(x, &ex);                /* |x| = m * 2^ex, 0.5 <= m < 1 */
    int lead = ex - 1;            /* position of the leading bit */
    int qexp = lead - 7;          /* 8 significant bits */
    if (qexp < -133)
        qexp = -133;              /* subnormal quantum */
    double q = ldexp(1.0, qexp);
    double r = nearbyint(x / q);  /* default rounding mode: ties to even */
    double y = r * q;
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(y) > bf16_max)
        return y > 0 ? 0x7F80 : 0xFF80;
    float fy = (float)y;          /* exact: y is a bf16 value */
    uint32_t u = f32_bits(fy);
    return (uint16_t)(u >> 16);
}

/*
 * E4M3 (the "fn" flavour: no infinities, NaN = S.1111.111): sign, 4 exponent
 * bits with bias 7, 3 mantissa bits.  Largest finite 1.75 * 2^8 = 448,
 * smallest normal 2^-6, subnormal quantum 2^-9.
 */
double oracle_e4m3_to_f64(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                 /* 0.mmm * 2^-6 */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);  /* 1.mmm * 2^(e-7) */
    return s ? -v : v;
}

/* Round to nearest even, saturating out-of-range finite values to +-448. */
uint8_t oracle_f64_to_e4m3_satfinite(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (isinf(a) || a >= 448.0) {
        /* anything at or beyond the largest finite value saturates */
        return (uint8_t)(sign | 0x7E);
    }
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);
    int lead = ex - 1;
    int qexp = lead - 3;          /* 4 significant bits */
    if (qexp < -9)
        qexp = -9;                /* subnormal quantum */
    double q = ldexp(1.0, qexp);
    double y = nearbyint(a / q) * q;
    if (y > 448.0)
        y = 448.0;                /* satfinite after rounding */
    if (y == 0.0)
        return sign;
    if (y < ldexp(1.0, -6)) {     /* subnormal: 0.mmm * 2^-6 */
        int m = (int)(y / ldexp(1.0, -9));
        return (uint8_t)(sign | m);
    }
    frexp(y, &ex);
    int e = ex - 1;               /* y = 1.f * 2^e exactly */
    int m = (int)((y / ldexp(1.0, e) - 1.0) * 8.0);
    return (uint8_t)(sign | ((e + 7) << 3) | m);
}

/*
 * The power-of-two block scale of [PithTrain] §7.2 (_compute_fp8_scale, the
 * non-e8m0 branch): t = fl32(max(fl32(amax), fl32(1e-4)) * fl32(1/448));
 * s = float with t's exponent field, bumped by one when t's mantissa is not
 * zero.  The product of two binary32 values is exact in binary64, so casting
 * it to float is the fp32 multiply.
 */
float oracle_fp8_block_scale(double amax)
{
    float a = (float)amax;
    float lo = (float)1e-4;
    float amax_clamped = a > lo ? a : lo;
    float rcp = (float)(1.0 / 448.0);
    float t = (float)((double)amax_clamped * (double)rcp);
    uint32_t bits = f32_bits(t);
    uint32_t mant = bits & 0x007FFFFFu;
    uint32_t sbits = (bits & 0x7F800000u) + (mant != 0 ? 0x00800000u : 0u);
    return f32_from_bits(sbits);
}

/*
 * The e8m0 branch of the same rule ([PithTrain] §7.2, _compute_fp8_scale with
 * SCALING_MODE "e8m0", the Blackwell path): the same fp32 product t, rounded
 * toward +infinity to a power of two 2^u, kept as the UE8M0 byte u + 127
 * (unsigned, 8 exponent bits, no mantissa; 0xFF is NaN), saturating at the
 * largest finite value 2^127 (byte 254).  The block scale is 2^(byte - 127).
 */
uint8_t oracle_ue8m0_block_scale(double amax)
{
    float a = (float)amax;
    float lo = (float)1e-4;
    float amax_clamped = a > lo ? a : lo;
    float rcp = (float)(1.0 / 448.0);
    double t = (double)(float)((double)amax_clamped * (double)rcp);
    if (isnan(t))
        return 0xFF;
    if (isinf(t))
        return 254;
    int ex;
    double m = frexp(t, &ex);          /* t = m * 2^ex, 0.5 <= m < 1 */
    int u = (m == 0.5) ? ex - 1 : ex;  /* smallest power of two >= t */
    int b = u + 127;
    if (b > 254)
        b = 254;
    if (b < 0)
        b = 0;
    return (uint8_t)b;
}

/* ------------------------------------------------------------------ */
/* Route  ([moe-engine] 融合Triton路由内核)                             */
/* ------------------------------------------------------------------ */

/*
 * For every token n:
 *   L[e]  = sum_h X[n,h] * W[h,e]  (+ bias[e])          -- fp64
 *   p[e]  = exp(L[e] - max L) / sum_e' exp(L[e'] - max L)
 *   top-K = K rounds of "largest remaining logit", strict '>' scanning e
 *           upwards (ties -> lower index), NaN treated as -inf
 *   w_k   = p[idx_k] / sum_j p[idx_j]   (renorm != 0)   else   w_k = p[idx_k]
 * X is bf16 [N,H], W is bf16 [H,E] (row-major, "tokens @ gate_w"), bias fp32
 * [E] or NULL.  topk_idx int32 [N,K], topk_w fp32 [N,K]; logits_out (fp64
 * [N,E]) and probs_out (fp64 [N,E]) are optional.
 */
int oracle_route(const uint16_t *X, const uint16_t *W, const float *bias,
                 int64_t N, int64_t H, int64_t E, int64_t K, int renorm,
                 int32_t *topk_idx, float *topk_w,
                 double *logits_out, double *probs_out)
{
    if (N < 0 || H <= 0 || E <= 0 || K <= 0 || K > E)
        return ORACLE_BAD_ARG;
    if (N == 0)
        return ORACLE_OK;
    int failed = 0;
#pragma omp parallel
    {
        double *L = (double *)malloc(sizeof(double) * (size_t)E);
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        char *chosen = (char *)malloc((size_t)E);
        if (!L || !p || !chosen) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t n = 0; n < N; ++n) {
                /* logits */
                for (int64_t e = 0; e < E; ++e)
                    L[e] = 0.0;
                for (int64_t h = 0; h < H; ++h) {
                    double x = oracle_bf16_to_f64(X[n * H + h]);
                    for (int64_t e = 0; e < E; ++e)
                        L[e] += x * oracle_bf16_to_f64(W[h * E + e]);
                }
                if (bias)
                    for (int64_t e = 0; e < E; ++e)
                        L[e] += (double)bias[e];
                /* softmax over all E experts */
                double m = -INFINITY;
                for (int64_t e = 0; e < E; ++e)
                    if (!isnan(L[e]) && L[e] > m)
                        m = L[e];
                double z = 0.0;
                for (int64_t e = 0; e < E; ++e) {
                    p[e] = isnan(L[e]) ? 0.0 : exp(L[e] - m);
                    z += p[e];
                }
                for (int64_t e = 0; e < E; ++e)
                    p[e] /= z;
                /* K rounds of selection */
                memset(chosen, 0, (size_t)E);
                double psel = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    int64_t best = -1;
                    double bestv = 0.0;
                    for (int64_t e = 0; e < E; ++e) {
                        if (chosen[e])
                            continue;
                        double v = isnan(L[e]) ? -INFINITY : L[e];
                        if (best < 0 || v > bestv) {
                            best = e;
                            bestv = v;
                        }
                    }
                    chosen[best] = 1;
                    topk_idx[n * K + k] = (int32_t)best;
                    psel += p[best];
                }
                /* weights */
                for (int64_t k = 0; k < K; ++k) {
                    double pk = p[topk_idx[n * K + k]];
                    topk_w[n * K + k] = (float)(renorm ? pk / psel : pk);
                }
                if (logits_out)
                    for (int64_t e = 0; e < E; ++e)
                        logits_out[n * E + e] = L[e];
                if (probs_out)
                    for (int64_t e = 0; e < E; ++e)
                        probs_out[n * E + e] = p[e];
            }
        }
        free(L);
        free(p);
        free(chosen);
    }
    return failed ? ORACLE_NO_MEM : ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Router statistics  ([moe-engine] 专家负载均衡)                       */
/* ------------------------------------------------------------------ */

/*
 * Per-token log-sum-exp of the router logits, the quantity a z-loss squares:
 * lse[n] = log( sum_e exp(L[n,e]) ), computed as m + log(sum_e exp(L[n,e] - m))
 * with m = max_e L[n,e], in fp64.  NaN logits count as -inf (as in the
 * selection); a token whose logits are all -inf gets -inf.
 * logits fp64 [N,E] (the logits_out of oracle_route), lse fp64 [N].
 */
int oracle_logsumexp(const double *logits, int64_t N, int64_t E, double *lse)
{
    if (N < 0 || E <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t n = 0; n < N; ++n) {
        double m = -INFINITY;
        for (int64_t e = 0; e < E; ++e) {
            double x = logits[n * E + e];
            if (!isnan(x) && x > m)
                m = x;
        }
        if (m == -INFINITY) {
            lse[n] = -INFINITY;
            continue;
        }
        double z = 0.0;
        for (int64_t e = 0; e < E; ++e) {
            double x = logits[n * E + e];
            if (!isnan(x))
                z += exp(x - m);
        }
        lse[n] = m + log(z);
    }
    return ORACLE_OK;
}

static int cmp_int32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * Expert-load statistics of the moe-engine page (section 专家负载均衡): the
 * imbalance ratio max/mean of the per-expert slot counts, the 95th percentile
 * of the counts over the mean, and the z-loss with weight coef:
 *   stats[0] = max_e counts[e] / mean,    mean = sum_e counts[e] / E
 *   stats[1] = P95(counts) / mean, P95 by linear interpolation between the
 *              sorted counts at position 0.95 * (E - 1)
 *   stats[2] = coef * (1/N) * sum_n lse[n]^2      (0 when lse is NULL or N == 0)
 *   stats[3] = mean
 * The ratios are 0 when no slot was counted.  All in fp64.
 */
int oracle_load_stats(const int32_t *counts, int64_t E, const double *lse, int64_t N,
                      double coef, double *stats)
{
    if (E <= 0 || N < 0)
        return ORACLE_BAD_ARG;
    int32_t *sorted = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!sorted)
        return ORACLE_NO_MEM;
    double total = 0.0, mx = 0.0;
    for (int64_t e = 0; e < E; ++e) {
        sorted[e] = counts[e];
        total += counts[e];
        if (counts[e] > mx)
            mx = counts[e];
    }
    qsort(sorted, (size_t)E, sizeof(int32_t), cmp_int32);
    double pos = 0.95 * (double)(E - 1);
    int64_t lo = (int64_t)floor(pos);
    int64_t hi = lo + 1 < E ? lo + 1 : E - 1;
    double p95 = sorted[lo] + (pos - (double)lo) * (double)(sorted[hi] - sorted[lo]);
    free(sorted);
    double mean = total / (double)E;
    stats[0] = mean > 0.0 ? mx / mean : 0.0;
    stats[1] = mean > 0.0 ? p95 / mean : 0.0;
    double zsum = 0.0;
    if (lse)
        for (int64_t n = 0; n < N; ++n)
            zsum += lse[n] * lse[n];
    stats[2] = (lse && N > 0) ? coef * zsum / (double)N : 0.0;
    stats[3] = mean;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Dispatch  ([PithTrain] §8.2, [moe-engine] Token守恒验证)             */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t expert;
    int64_t slot;
} slot_key;

static int cmp_slot_key(const void *a, const void *b)
{
    const slot_key *x = (const slot_key *)a;
    const slot_key *y = (const slot_key *)b;
    if (x->expert != y->expert)
        return x->expert < y->expert ? -1 : 1;
    if (x->slot != y->slot)
        return x->slot < y->slot ? -1 : 1;
    return 0;
}

/*
 * counts[e]   = number of slots (n,k) with topk_idx[n*K+k] == e
 * offsets[e]  = sum_{e' < e} counts[e'],  offsets[E] = N*K
 * row_map[s]  = rank of slot s in the order (expert, s): the stable argsort
 *               of the slots by expert (a total order, so the result is
 *               unique; sorting the (expert, slot) pairs gives it directly)
 * src_slot[r] = the slot whose row is r (inverse of row_map); may be NULL.
 * Returns ORACLE_BAD_INDEX if an index is outside [0,E).
 */
int oracle_dispatch(const int32_t *topk_idx, int64_t N, int64_t E, int64_t K,
                    int32_t *counts, int32_t *offsets, int32_t *row_map,
                    int32_t *src_slot)
{
    if (N < 0 || E <= 0 || K <= 0)
        return ORACLE_BAD_ARG;
    int64_t S = N * K;
    for (int64_t s = 0; s < S; ++s)
        if (topk_idx[s] < 0 || topk_idx[s] >= E)
            return ORACLE_BAD_INDEX;
    for (int64_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t s = 0; s < S; ++s)
        counts[topk_idx[s]] += 1;
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    if (S == 0)
        return ORACLE_OK;
    slot_key *keys = (slot_key *)malloc(sizeof(slot_key) * (size_t)S);
    if (!keys)
        return ORACLE_NO_MEM;
    for (int64_t s = 0; s < S; ++s) {
        keys[s].expert = topk_idx[s];
        keys[s].slot = s;
    }
    qsort(keys, (size_t)S, sizeof(slot_key), cmp_slot_key);
    for (int64_t r = 0; r < S; ++r) {
        row_map[keys[r].slot] = (int32_t)r;
        if (src_slot)
            src_slot[r] = (int32_t)keys[r].slot;
    }
    free(keys);
    return ORACLE_OK;
}

/*
 * Expert-parallel dispatch metadata with token deduplication ([PithTrain]
 * §8.2, fused_dedup_prepare_dispatch: per-expert and per-EP-rank counts,
 * prefix sums, send metadata, dedup scatter, counting sort and expand_idx),
 * for the tokens of one GPU.  Experts are split over R = ep_size ranks,
 * P = E / R consecutive experts each: rank(e) = e / P.  A token goes to a
 * rank once however many of its K experts live there (deduplication).
 *   rank_counts[r]   = #{n : some k has rank(topk[n,k]) == r}
 *   rank_offsets[r]  = sum_{r' < r} rank_counts[r'],  rank_offsets[R] = total rows
 *   send_token[row]  = the token of send row `row`; rows are ordered by
 *                      (rank, token): rank-contiguous, tokens ascending
 *   slot_send_row[s] = the send row carrying the token of slot s to the rank
 *                      of its expert
 *   expand_idx[row]  = for row `row` of the expert-contiguous order of
 *                      oracle_dispatch (slot s = its src_slot), the index of
 *                      s's token within its rank's block of send rows:
 *                      slot_send_row[s] - rank_offsets[rank(topk[s])]
 *   send_meta[r*(P+1)]         = rank_counts[r]
 *   send_meta[r*(P+1) + 1 + j] = counts[r*P + j]   (the per-rank metadata
 *                      exchanged before the token all-to-all, dedup count first)
 * counts / offsets / row_map / src_slot as in oracle_dispatch.  send_token is
 * sized for N * min(K, R) rows.  Returns ORACLE_BAD_ARG unless E % R == 0.
 */
int oracle_dispatch_ep(const int32_t *topk_idx, int64_t N, int64_t E, int64_t K, int64_t R,
                       int32_t *counts, int32_t *offsets, int32_t *row_map, int32_t *src_slot,
                       int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_token,
                       int32_t *slot_send_row, int32_t *expand_idx, int32_t *send_meta)
{
    if (N < 0 || E <= 0 || K <= 0 || R <= 0 || E % R != 0)
        return ORACLE_BAD_ARG;
    int st = oracle_dispatch(topk_idx, N, E, K, counts, offsets, row_map, src_slot);
    if (st != ORACLE_OK)
        return st;
    int64_t P = E / R;
    /* row of (rank r, token n), -1 if the token has no expert on r */
    int32_t *row_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R * (N > 0 ? N : 1)));
    if (!row_of)
        return ORACLE_NO_MEM;
    int32_t row = 0;
    for (int64_t r = 0; r < R; ++r) {
        rank_offsets[r] = row;
        for (int64_t n = 0; n < N; ++n) {
            int hit = 0;
            for (int64_t k = 0; k < K; ++k)
                if (topk_idx[n * K + k] / P == r)
                    hit = 1;
            row_of[r * N + n] = hit ? row : -1;
            if (hit)
                send_token[row++] = (int32_t)n;
        }
        rank_counts[r] = row - rank_offsets[r];
    }
    rank_offsets[R] = row;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            slot_send_row[n * K + k] = row_of[(topk_idx[n * K + k] / P) * N + n];
    for (int64_t q = 0; q < N * K; ++q) {
        int64_t s = src_slot[q];
        int64_t r = topk_idx[s] / P;
        expand_idx[q] = slot_send_row[s] - rank_offsets[r];
    }
    for (int64_t r = 0; r < R; ++r) {
        send_meta[r * (P + 1)] = rank_counts[r];
        for (int64_t j = 0; j < P; ++j)
            send_meta[r * (P + 1) + 1 + j] = counts[r * P + j];
    }
    free(row_of);
    return ORACLE_OK;
}

/*
 * Xp[row_map[n*K+k], :] = X[n, :]   (bf16 bits copied)
 * If Xq/Xs are given (H % 128 == 0), every 1x128 block b of X[n,:] also
 * gives s = oracle_fp8_block_scale(max |x|) and q = E4M3(x / s); both are
 * written to each of the token's K destination rows:
 * Xq [N*K, H] (one byte per element), Xs [N*K, H/128] fp32.
 */
int oracle_permute(const uint16_t *X, const int32_t *row_map,
                   int64_t N, int64_t H, int64_t K,
                   uint16_t *Xp, uint8_t *Xq, float *Xs)
{
    if (N < 0 || H <= 0 || K <= 0)
        return ORACLE_BAD_ARG;
    if ((Xq || Xs) && (H % 128 != 0 || !Xq || !Xs))
        return ORACLE_BAD_ARG;
    int64_t nb = H / 128;
    for (int64_t s = 0; s < N * K; ++s)
        if (row_map[s] < 0 || row_map[s] >= N * K)
            return ORACLE_BAD_INDEX;
    /* tokens are independent (each destination row has one source slot) */
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t r = row_map[n * K + k];
            if (Xp)
                memcpy(Xp + r * H, X + n * H, sizeof(uint16_t) * (size_t)H);
            if (Xq) {
                for (int64_t b = 0; b < nb; ++b) {
                    double amax = 0.0;
                    for (int64_t j = 0; j < 128; ++j) {
                        double v = fabs(oracle_bf16_to_f64(X[n * H + b * 128 + j]));
                        if (v > amax)
                            amax = v;
                    }
                    float s = oracle_fp8_block_scale(amax);
                    Xs[r * nb + b] = s;
                    for (int64_t j = 0; j < 128; ++j) {
                        double x = oracle_bf16_to_f64(X[n * H + b * 128 + j]);
                        Xq[r * H + b * 128 + j] = oracle_f64_to_e4m3_satfinite(x / (double)s);
                    }
                }
            }
        }
    }
    return ORACLE_OK;
}

/*
 * The E4M3 copy of the permute with UE8M0 block scales (the e8m0 branch):
 * for every 1x128 block b of X[n,:], byte = oracle_ue8m0_block_scale(max |x|),
 * s = 2^(byte - 127), q = E4M3(x / s); both written to each of the token's K
 * destination rows.  Xq [N*K, H], Xs8 [N*K, H/128] one byte per block.
 */
int oracle_permute_ue8m0(const uint16_t *X, const int32_t *row_map,
                         int64_t N, int64_t H, int64_t K,
                         uint8_t *Xq, uint8_t *Xs8)
{
    if (N < 0 || H <= 0 || K <= 0 || H % 128 != 0 || !Xq || !Xs8)
        return ORACLE_BAD_ARG;
    int64_t nb = H / 128;
    for (int64_t s = 0; s < N * K; ++s)
        if (row_map[s] < 0 || row_map[s] >= N * K)
            return ORACLE_BAD_INDEX;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t r = row_map[n * K + k];
            for (int64_t b = 0; b < nb; ++b) {
                double amax = 0.0;
                for (int64_t j = 0; j < 128; ++j) {
                    double v = fabs(oracle_bf16_to_f64(X[n * H + b * 128 + j]));
                    if (v > amax)
                        amax = v;
                }
                uint8_t e = oracle_ue8m0_block_scale(amax);
                double sc = ldexp(1.0, (int)e - 127);
                Xs8[r * nb + b] = e;
                for (int64_t j = 0; j < 128; ++j) {
                    double x = oracle_bf16_to_f64(X[n * H + b * 128 + j]);
                    Xq[r * H + b * 128 + j] = oracle_f64_to_e4m3_satfinite(x / sc);
                }
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Combine  ([PithTrain] §6.1 forward_aggregate, weighted part)         */
/* ------------------------------------------------------------------ */

/*
 * out[n,h] = bf16_rne( sum_{k=0}^{K-1} w[n,k] * Y[row_map[n*K+k], h] )
 * with the sum in fp64.  Y bf16 [N*K, H], w fp32 [N,K], out bf16 [N,H].
 */
int oracle_combine(const uint16_t *Y, const int32_t *row_map, const float *w,
                   int64_t N, int64_t H, int64_t K, uint16_t *out)
{
    if (N < 0 || H <= 0 || K <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t s = 0; s < N * K; ++s)
        if (row_map[s] < 0 || row_map[s] >= N * K)
            return ORACLE_BAD_INDEX;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t r = row_map[n * K + k];
                acc += (double)w[n * K + k] * oracle_bf16_to_f64(Y[r * H + h]);
            }
            out[n * H + h] = oracle_f64_to_bf16(acc);
        }
    }
    return ORACLE_OK;
}

/*
 * Combine with the residual connection: the whole of forward_aggregate
 * ([PithTrain] §6.1, "weighted expert output + residual connection"):
 * out[n,h] = bf16_rne( sum_{k=0}^{K-1} w[n,k] * Y[row_map[n*K+k], h] + residual[n,h] )
 * with the weighted sum and the addition in fp64 and one rounding at the end.
 * residual bf16 [N,H].
 */
int oracle_combine_residual(const uint16_t *Y, const int32_t *row_map, const float *w,
                            const uint16_t *residual, int64_t N, int64_t H, int64_t K,
                            uint16_t *out)
{
    if (N < 0 || H <= 0 || K <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t s = 0; s < N * K; ++s)
        if (row_map[s] < 0 || row_map[s] >= N * K)
            return ORACLE_BAD_INDEX;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t r = row_map[n * K + k];
                acc += (double)w[n * K + k] * oracle_bf16_to_f64(Y[r * H + h]);
            }
            acc += oracle_bf16_to_f64(residual[n * H + h]);
            out[n * H + h] = oracle_f64_to_bf16(acc);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Synthetic expert outputs for the combine step                       */
/* ------------------------------------------------------------------ */

/*
 * Stand-in for the expert MLP (which is outside the routing path): row p of
 * the expert-contiguous buffer, owned by expert e(p) (offsets[e] <= p <
 * offsets[e+1]), becomes Y[p,h] = bf16_rne(fl32(Xp[p,h] * fl32(1 + e/E))).
 * The product is formed in fp32 and rounded once more to bf16, so that a
 * float32 tensor library computing the same fixture gets the same bits.
 */
int oracle_expert_fixture(const uint16_t *Xp, const int32_t *offsets,
                          int64_t E, int64_t rows, int64_t H, uint16_t *Y)
{
    if (E <= 0 || rows < 0 || H <= 0 || offsets[E] != rows)
        return ORACLE_BAD_ARG;
    for (int64_t e = 0; e < E; ++e) {
        float f = (float)(1.0 + (double)e / (double)E);
#pragma omp parallel for schedule(static)
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p)
            for (int64_t h = 0; h < H; ++h) {
                double x = oracle_bf16_to_f64(Xp[p * H + h]);
                float prod = (float)(x * (double)f);
                Y[p * H + h] = oracle_f64_to_bf16((double)prod);
            }
    }
    return ORACLE_OK;
}

/* Host threads the OpenMP loops above use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the threads of the OpenMP loops (n >= 1); no effect without OpenMP. */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
