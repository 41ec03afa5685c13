/*
 * moe_oracle.c -- plain, slow CPU reference for the Mixture-of-Experts
 * routing / dispatch-planning hot path (route top-k, plan, permute, combine).
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the smoke check and the CPU
 * baseline leg of the benchmark load this file; the product library never
 * does, and this file includes nothing from it.
 *
 * Every function is the plain definition of its step, written as loops in
 * the order the sources give, with no blocking, fusion or reordering.
 * Sources (by page title and section):
 *   [MoonEP]  MoonEP, moonep/planning.py: PlanningKernel (run_c1 histogram /
 *             prefix / stable scatter; per-rank cu_seqlens and
 *             zero_fill_ranges; dst computation; duplicate canonicalisation;
 *             src_info provenance) and the MoonEPCommPlan record.
 *   [TRT]     TensorRT-LLM, trtllmGenKernels/blockScaleMoe/RoutingKernel.cuh:
 *             calcSoftmax (full and top-K variants), sigmoid_accurate,
 *             routingPermutation / routingIndicesOffsetsKernel.
 *   [DeepEP]  DeepEP, csrc/kernels/intranode.cu: notify_dispatch (rank
 *             prefix matrix, aligned per-expert counts), dispatch (row
 *             copy), combine (fp32 accumulation, cast back to the dtype).
 * Where the sources are silent the reading taken is named in a comment
 * ("reading: ...").
 *
 * Floating point: the router weights are computed in fp64 (the exact
 * value the fp32 GPU result is compared against).  Two places decide an
 * integer from floating point and therefore fix fp32: the selection key of
 * the sigmoid router (sigmoid + correction bias, and the group score) and
 * the fp32 accumulation of the combine, whose precision DeepEP's combine
 * fixes (fp32 accumulate, cast to bf16).  Compile with -ffp-contract=off
 * and without fast-math so every operation below rounds exactly once.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_EUNSUP 2
#define ORC_ECAP 3

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32                                                       */
/* ------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32: widening is exact. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to bf16, nearest with ties to even.  NaN inputs are
 * outside the contract of the combine (inputs are finite); they map to a
 * quiet NaN of the same sign. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* fp32 exponential and sigmoid by one fixed operation sequence          */
/* ------------------------------------------------------------------ */
/*
 * The sigmoid router ranks experts by sigmoid(logit) + bias in fp32.  The
 * pages define sigmoid as 0.5*tanh(0.5x)+0.5 (TRT, sigmoid_accurate) but
 * name no tanh/exp implementation, and libm results differ by an ulp
 * between libraries, which would flip top-k boundaries.  Reading: the
 * selection key uses sigmoid(x) = 1/(1+e^-x) (the same function), with
 * e^t (t <= 0) evaluated by Cody & Waite's argument reduction
 * t = n*ln2 + r, |r| <= ln2/2, ln2 split into a 16-significant-bit head
 * (exact products n*ln2_hi for |n| <= 256) and an fp32 tail, followed by
 * the degree-7 Taylor polynomial of e^r (coefficients 1/j!) in Horner form
 * with one fused multiply-add per step, then scaling by 2^n in two exact
 * power-of-two factors.  Truncation error r^8/8! <= 5.3e-9 relative.
 */
static float pow2_int(int n) /* 2^n, -126 <= n <= 127 */
{
    uint32_t u = (uint32_t)(n + 127) << 23;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float orc_exp_f32(float t) /* defined for t <= 0 (the only use) */
{
    if (t != t)
        return t;
    if (t > 0.0f)
        t = 0.0f; /* reading: callers only pass t <= 0; clamp keeps n <= 0 */
    if (t < -104.0f)
        return 0.0f; /* e^t < 2^-150: rounds to zero */
    const float log2e = (float)1.4426950408889634;   /* 1/ln 2 */
    const float ln2_hi = 0.693145751953125f;          /* ln 2 to 16 bits */
    const float ln2_lo = (float)(0.6931471805599453 - 0.693145751953125);
    float nf = rintf(t * log2e);                      /* nearest, ties even */
    float r = fmaf(-nf, ln2_hi, t);
    r = fmaf(-nf, ln2_lo, r);
    float p = (float)(1.0 / 5040.0);
    p = fmaf(p, r, (float)(1.0 / 720.0));
    p = fmaf(p, r, (float)(1.0 / 120.0));
    p = fmaf(p, r, (float)(1.0 / 24.0));
    p = fmaf(p, r, (float)(1.0 / 6.0));
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int n = (int)nf;      /* -150 <= n <= 0 */
    int n1 = n / 2;       /* truncates toward zero */
    int n2 = n - n1;
    return (p * pow2_int(n1)) * pow2_int(n2);
}

float orc_sigmoid_f32(float x)
{
    if (x != x)
        return x;
    if (x >= 0.0f) {
        float e = orc_exp_f32(-x);
        return 1.0f / (1.0f + e);
    }
    float e = orc_exp_f32(x);
    return e / (1.0f + e);
}

/* ------------------------------------------------------------------ */
/* Router: scores, (group-limited) top-K, weights                        */
/* ------------------------------------------------------------------ */
/*
 * scoring 0 (softmax, TRT calcSoftmax): selection key = the fp32 logit
 *   (softmax is strictly increasing, so ranking logits ranks
 *   probabilities).  renormalize=1: w_k = exp(l_k - l_max) /
 *   sum_{j in top-K} exp(l_j - l_max) (the top-K-lane calcSoftmax);
 *   renormalize=0: the denominator runs over all E experts.
 * scoring 1 (sigmoid): s_e = sigmoid(l_e); key_e = s_e + bias_e (fp32).
 *   Optional group-limited selection (reading, DeepSeek-V3 style routing
 *   that the pages reference but do not show): the E experts form
 *   n_group contiguous groups; a group's score is the fp32 sum of its two
 *   largest keys (its only key when a group has one expert); the
 *   topk_group best groups are kept; top-K runs over their experts.
 *   Weights use the unbiased scores: w_k = s_k / sum_j s_j
 *   (renormalize=1) or s_k (renormalize=0).
 * All weights are multiplied by routed_scaling.
 * Order: descending key; equal keys go to the lower index first (MoonEP
 * warp_argmax_min_idx: value by max, tie broken by the minimum index).
 * The same rule ranks groups.
 */
static int argmax_lowest(const float* key, const unsigned char* usable, int n)
{
    int best = -1;
    for (int e = 0; e < n; ++e) {
        if (!usable[e])
            continue;
        if (best < 0 || key[e] > key[best])
            best = e;
    }
    return best;
}

int orc_route_topk(const float* logits, const float* bias, int N, int E, int K,
                   int scoring, int renormalize, int n_group, int topk_group,
                   float routed_scaling, int32_t* topk_idx, double* topk_w)
{
    if (N < 0 || E < 1 || K < 1 || K > E || K > 32)
        return ORC_EINVAL;
    if (scoring != 0 && scoring != 1)
        return ORC_EINVAL;
    if (n_group < 1)
        return ORC_EINVAL;
    if (n_group > 1) {
        if (scoring != 1)
            return ORC_EUNSUP;
        if (E % n_group != 0 || topk_group < 1 || topk_group > n_group ||
            K > topk_group * (E / n_group))
            return ORC_EINVAL;
    }
    if (bias && scoring != 1)
        return ORC_EUNSUP;

    float* key = (float*)malloc(sizeof(float) * (size_t)E);
    unsigned char* usable = (unsigned char*)malloc((size_t)E);
    float* gscore = (float*)malloc(sizeof(float) * (size_t)n_group);
    unsigned char* gusable = (unsigned char*)malloc((size_t)n_group);
    unsigned char* gkept = (unsigned char*)malloc((size_t)n_group);
    if (!key || !usable || !gscore || !gusable || !gkept) {
        free(key); free(usable); free(gscore); free(gusable); free(gkept);
        return ORC_ECAP;
    }

    for (int s = 0; s < N; ++s) {
        const float* l = logits + (size_t)s * E;
        for (int e = 0; e < E; ++e) {
            if (scoring == 0)
                key[e] = l[e];
            else {
                float sg = orc_sigmoid_f32(l[e]);
                key[e] = bias ? sg + bias[e] : sg;
            }
            usable[e] = 1;
        }

        if (n_group > 1) {
            int gs = E / n_group;
            for (int g = 0; g < n_group; ++g) {
                const float* gk = key + (size_t)g * gs;
                int i1 = 0;
                for (int j = 1; j < gs; ++j)
                    if (gk[j] > gk[i1])
                        i1 = j;
                if (gs == 1) {
                    gscore[g] = gk[i1];
                } else {
                    int i2 = -1;
                    for (int j = 0; j < gs; ++j) {
                        if (j == i1)
                            continue;
                        if (i2 < 0 || gk[j] > gk[i2])
                            i2 = j;
                    }
                    gscore[g] = gk[i1] + gk[i2];
                }
                gusable[g] = 1;
                gkept[g] = 0;
            }
            for (int r = 0; r < topk_group; ++r) {
                int g = argmax_lowest(gscore, gusable, n_group);
                gkept[g] = 1;
                gusable[g] = 0;
            }
            for (int e = 0; e < E; ++e)
                usable[e] = gkept[e / gs];
        }

        int32_t* idx = topk_idx + (size_t)s * K;
        for (int k = 0; k < K; ++k) {
            int e = argmax_lowest(key, usable, E);
            idx[k] = e;
            usable[e] = 0;
        }

        double* w = topk_w + (size_t)s * K;
        if (scoring == 0) {
            double m = (double)l[idx[0]]; /* top-1 logit = the row maximum */
            double denom = 0.0;
            if (renormalize) {
                for (int k = 0; k < K; ++k)
                    denom += exp((double)l[idx[k]] - m);
            } else {
                for (int e = 0; e < E; ++e)
                    denom += exp((double)l[e] - m);
            }
            for (int k = 0; k < K; ++k)
                w[k] = exp((double)l[idx[k]] - m) / denom * (double)routed_scaling;
        } else {
            double denom = 0.0;
            for (int k = 0; k < K; ++k)
                denom += 1.0 / (1.0 + exp(-(double)l[idx[k]]));
            for (int k = 0; k < K; ++k) {
                double sk = 1.0 / (1.0 + exp(-(double)l[idx[k]]));
                w[k] = (renormalize ? sk / denom : sk) * (double)routed_scaling;
            }
        }
    }

    free(key); free(usable); free(gscore); free(gusable); free(gkept);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Dispatch plan                                                        */
/* ------------------------------------------------------------------ */

/* Rows the caller provides for the permuted buffer: every pair plus the
 * worst-case alignment padding of every expert. */
int64_t orc_plan_capacity_rows(int N, int E, int K, int alignment)
{
    return (int64_t)N * K + (int64_t)E * (alignment - 1);
}

/*
 * Inputs: topk[N*K] expert ids, flat pair index f = s*K + k.
 * Logical rank r owns experts [r*epn, (r+1)*epn), epn = E/R (MoonEP dst
 * computation: owner rank = expert / epn; DeepEP notify_dispatch: the
 * per-rank expert block).
 *
 *  1. count_e = #{f : topk[f] = e}                      (MoonEP run_c1 1a;
 *     TRT routingIndicesHistogramKernel)
 *  2. padded_e = count_e > 0 ? ceil(count_e / a) * a : 0 (MoonEP per-rank
 *     cu_seqlens; DeepEP aligned receive counts)
 *     cu[0] = 0, cu[e+1] = cu[e] + padded_e.  Reading: one global
 *     expert-major buffer with a leading zero; MoonEP's rank-local padded
 *     ends are cu[e+1] - cu[r*epn].
 *  3. zero_fill[e] = (cu[e] + count_e, padded_e - count_e) when the
 *     padding is positive, else (0, 0)                   (MoonEP)
 *  4. raw slot(f) = cu[e] + #{f' < f : topk[f'] = e}: within an expert,
 *     pairs keep ascending flat index (MoonEP run_c1 pass A, the stable
 *     scatter into `order`).  Reading: the slot is global (the rank-strided
 *     rank*NvS + loff of one GPU maps one-to-one onto it).
 *  5. dst[f] = raw slot when f is the first pair of its token on its
 *     rank (k ascending), else -raw-1                   (MoonEP duplicate
 *     canonicalisation)
 *  6. src_of_slot[raw slot(f)] = f, every other row of the P_cap rows -1
 *     (MoonEP src_info, -1 for an empty slot)
 *  7. is_token_in_rank[s*R + r], tokens_per_rank[r] = #tokens with a pair
 *     on r, pairs_per_rank[r] = sum of counts of r's experts,
 *     rank_prefix[0] = 0, rank_prefix[r+1] = rank_prefix[r] +
 *     tokens_per_rank[r] (DeepEP notify_dispatch with one source rank),
 *     rank_slot_offsets[r] = cu[r*epn] for r = 0..R.
 *  8. Reading (the dispatch builder that fills these is not on the pages,
 *     and its order is atomic): one group per (token, rank) holding >= 2
 *     pairs, ordered by (token, first k).  dup_groups[g] = (primary raw
 *     slot, dup_begin, dup_count); dup_loffs[dup_begin + i] = raw slot of
 *     the group's i-th duplicate in k order; dup_counts = (groups, dups).
 */
int orc_plan(const int32_t* topk, int N, int E, int K, int R, int alignment,
             int32_t* tokens_per_expert, int32_t* cu_seqlens, int32_t* zero_fill_ranges,
             int32_t* pairs_per_rank, int32_t* tokens_per_rank, int32_t* rank_prefix,
             int32_t* rank_slot_offsets, uint8_t* is_token_in_rank, int32_t* dst,
             int32_t* src_of_slot, int64_t src_capacity,
             int32_t* dup_groups, int64_t group_capacity,
             int32_t* dup_loffs, int64_t dup_capacity, int32_t* dup_counts)
{
    if (N < 0 || E < 1 || K < 1 || R < 1 || alignment < 1 || E % R != 0)
        return ORC_EINVAL;
    if (src_capacity < orc_plan_capacity_rows(N, E, K, alignment))
        return ORC_ECAP;
    const int epn = E / R;
    const int64_t NK = (int64_t)N * K;
    for (int64_t f = 0; f < NK; ++f)
        if (topk[f] < 0 || topk[f] >= E)
            return ORC_EINVAL;

    /* 1. histogram */
    for (int e = 0; e < E; ++e)
        tokens_per_expert[e] = 0;
    for (int64_t f = 0; f < NK; ++f)
        tokens_per_expert[topk[f]] += 1;

    /* 2. aligned exclusive scan; 3. zero-fill ranges */
    cu_seqlens[0] = 0;
    for (int e = 0; e < E; ++e) {
        int32_t c = tokens_per_expert[e];
        int32_t padded = c > 0 ? (int32_t)(((int64_t)c + alignment - 1) / alignment * alignment) : 0;
        cu_seqlens[e + 1] = cu_seqlens[e] + padded;
        if (padded - c > 0) {
            zero_fill_ranges[2 * e] = cu_seqlens[e] + c;
            zero_fill_ranges[2 * e + 1] = padded - c;
        } else {
            zero_fill_ranges[2 * e] = 0;
            zero_fill_ranges[2 * e + 1] = 0;
        }
    }

    /* 4. stable slots (running count per expert, pairs in f order) and
     * 6. provenance */
    int32_t* seen = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    int32_t* raw = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NK > 0 ? NK : 1));
    if (!seen || !raw) {
        free(seen); free(raw);
        return ORC_ECAP;
    }
    for (int64_t i = 0; i < src_capacity; ++i)
        src_of_slot[i] = -1;
    for (int64_t f = 0; f < NK; ++f) {
        int e = topk[f];
        raw[f] = cu_seqlens[e] + seen[e];
        seen[e] += 1;
        src_of_slot[raw[f]] = (int32_t)f;
    }

    /* 5. duplicate canonicalisation and 7. rank membership */
    for (int r = 0; r < R; ++r) {
        tokens_per_rank[r] = 0;
        pairs_per_rank[r] = 0;
    }
    for (int e = 0; e < E; ++e)
        pairs_per_rank[e / epn] += tokens_per_expert[e];
    for (int s = 0; s < N; ++s) {
        uint8_t* row = is_token_in_rank + (size_t)s * R;
        for (int r = 0; r < R; ++r)
            row[r] = 0;
        for (int k = 0; k < K; ++k) {
            int64_t f = (int64_t)s * K + k;
            int r = topk[f] / epn;
            dst[f] = row[r] ? -raw[f] - 1 : raw[f];
            row[r] = 1;
        }
        for (int r = 0; r < R; ++r)
            tokens_per_rank[r] += row[r];
    }
    rank_prefix[0] = 0;
    for (int r = 0; r < R; ++r)
        rank_prefix[r + 1] = rank_prefix[r] + tokens_per_rank[r];
    for (int r = 0; r <= R; ++r)
        rank_slot_offsets[r] = cu_seqlens[r * epn];

    /* 8. dedup structures, groups in (token, first k) order */
    int64_t n_groups = 0, n_dup = 0;
    int rc = ORC_OK;
    for (int s = 0; s < N && rc == ORC_OK; ++s) {
        for (int k = 0; k < K; ++k) {
            int64_t f = (int64_t)s * K + k;
            if (dst[f] < 0)
                continue; /* only a primary opens a group */
            int r = topk[f] / epn;
            int later = 0;
            for (int k2 = k + 1; k2 < K; ++k2)
                if (topk[(int64_t)s * K + k2] / epn == r)
                    later += 1;
            if (later == 0)
                continue;
            if (n_groups >= group_capacity || n_dup + later > dup_capacity) {
                rc = ORC_ECAP;
                break;
            }
            dup_groups[3 * n_groups + 0] = raw[f];
            dup_groups[3 * n_groups + 1] = (int32_t)n_dup;
            dup_groups[3 * n_groups + 2] = later;
            n_groups += 1;
            for (int k2 = k + 1; k2 < K; ++k2)
                if (topk[(int64_t)s * K + k2] / epn == r)
                    dup_loffs[n_dup++] = raw[(int64_t)s * K + k2];
        }
    }
    dup_counts[0] = (int32_t)n_groups;
    dup_counts[1] = (int32_t)n_dup;

    free(seen);
    free(raw);
    return rc;
}

/* ------------------------------------------------------------------ */
/* Permute and combine                                                  */
/* ------------------------------------------------------------------ */

/* Decode a dst entry to its raw slot (MoonEP: duplicates carry -raw-1). */
static int32_t raw_slot(int32_t d)
{
    return d >= 0 ? d : -d - 1;
}

/*
 * permuted[raw slot(f)] = x[f / K] bit for bit, for every pair (primary
 * and duplicate: each expert needs its own row); rows inside the
 * zero-fill ranges are +0.0.  Rows at or beyond cu[E] are not written.
 * (DeepEP dispatch copies a token's hidden row; MoonEP names the padded
 * ranges.  Reading: the permute writes the padding zeros itself.)
 */
void orc_permute(const uint16_t* x, int N, int H, int K, const int32_t* dst,
                 const int32_t* zero_fill_ranges, int E, uint16_t* permuted)
{
    for (int64_t f = 0; f < (int64_t)N * K; ++f) {
        int64_t s = f / K;
        int64_t row = raw_slot(dst[f]);
        memcpy(permuted + row * H, x + s * H, sizeof(uint16_t) * (size_t)H);
    }
    for (int e = 0; e < E; ++e) {
        int64_t start = zero_fill_ranges[2 * e];
        int64_t count = zero_fill_ranges[2 * e + 1];
        for (int64_t j = 0; j < count; ++j)
            memset(permuted + (start + j) * H, 0, sizeof(uint16_t) * (size_t)H);
    }
}

/*
 * out[s, h] = bf16_rne( acc ), acc = 0; for k = 0..K-1:
 *     acc = fmaf(w[s,k], float(y[raw slot(s,k), h]), acc).
 * DeepEP's combine accumulates the rows in fp32 and casts back to bf16;
 * reading: the weighted form, with the weight applied by one fused
 * multiply-add per pair in k order.
 */
void orc_combine(const uint16_t* y, const float* w, const int32_t* dst,
                 int N, int K, int H, uint16_t* out)
{
    for (int64_t s = 0; s < N; ++s) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t f = s * K + k;
                int64_t row = raw_slot(dst[f]);
                acc = fmaf(w[f], orc_bf16_to_f32(y[row * H + h]), acc);
            }
            out[s * H + h] = orc_f32_to_bf16(acc);
        }
    }
}

/* The same combine for a list of tokens only (spot checks at full size). */
void orc_combine_rows(const uint16_t* y, const float* w, const int32_t* dst,
                      const int64_t* tokens, int n_tokens, int K, int H, uint16_t* out)
{
    for (int i = 0; i < n_tokens; ++i) {
        int64_t s = tokens[i];
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t f = s * K + k;
                int64_t row = raw_slot(dst[f]);
                acc = fmaf(w[f], orc_bf16_to_f32(y[row * H + h]), acc);
            }
            out[(int64_t)i * H + h] = orc_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Capacity-balanced plan with redundant experts                       */
/* ------------------------------------------------------------------ */
/*
 * MoonEP moonep/planning.py, PlanningKernel, the rank-0 planning steps and
 * the dst computation, in their single-source form (one GPU holds every
 * token, so the prefix over source ranks of tokens per expert is just the
 * expert's count).  Steps, in the page's order:
 *
 *  S1  group_tokens[r] = pairs routed to rank r's experts.
 *  Balance: balance[r] = group_tokens[r] - CAP.  While some rank has
 *      balance > 0 and some < 0: surplus = the largest balance, deficit =
 *      the smallest (ties: lower rank); move = -deficit tokens from the
 *      surplus rank to the deficit rank: z[surplus][deficit] = move,
 *      balance[surplus] -= move, balance[deficit] = 0.  Each step zeroes one
 *      rank and a zeroed rank never moves again, so at most R steps.
 *  Alloc (per owner rank o): quotas[r] = z[o][r]; remaining[le] = count of
 *      o's le-th expert.  While the largest quota (ties: lower rank) and
 *      the largest remaining count (ties: lower expert) are both positive:
 *      take = min of the two; that many of the expert's pairs go to the
 *      quota rank.  alloc[r][e] = pairs of expert e handled by rank r
 *      (its owner keeps the rest); alloc_cumsum[e][r] = inclusive prefix
 *      over r.
 *  Selection (per destination rank d): remote[e] = alloc[d][e] for experts
 *      not owned by d, else 0; remote_stats[d][0] = #{e : remote[e] > 0}.
 *      B rounds: pick the largest remote count, ties to the HIGHER expert
 *      index (the page's ">=" scan); experts_to_copy[d][slot] = that expert
 *      if its count > 0, else -1; the pick is cleared; a real pick adds 1
 *      to remote_stats[owner][1].
 *  Groups g in [0, E+B) of rank d: g < E holds expert g with count
 *      alloc[d][g] unless g was picked (then 0); g >= E holds the expert of
 *      slot g-E with count alloc[d][that expert] (0 for -1).
 *      padded = round_up(count, tp) if count > 0 else 0; base = exclusive
 *      prefix of padded over g; cu_seqlens[d][g] = base + padded (padded
 *      end, rank-local); zero_fill[d][g] = (base + count, padded - count)
 *      when count > 0 and padded > count, else (0, 0); expert_offsets[d][e]
 *      = base of the group holding expert e when its count > 0.  Reading:
 *      entries the page leaves unwritten are 0.
 *  dst: for pair f of expert e at position gr among e's pairs (ascending
 *      flat index), the destination rank is the first r with
 *      alloc_cumsum[e][r] > gr; pc = alloc_cumsum[e][r-1] (0 for r = 0);
 *      dst[f] = r * NvS + expert_offsets[r][e] + (gr - pc).  Then the
 *      duplicate canonicalisation by destination rank (dst / NvS), as in
 *      the plain plan: a later pair of a token on an already-seen rank
 *      stores -dst-1.
 * Returns ORC_ECAP when a rank's groups need more than NvS rows.
 */
static int argmax_low_i32(const int32_t* v, int n) /* largest value, lowest index */
{
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best])
            best = i;
    return best;
}

static int argmin_low_i32(const int32_t* v, int n) /* smallest value, lowest index */
{
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] < v[best])
            best = i;
    return best;
}

int orc_plan_balanced(const int32_t* topk, int N, int E, int K, int R, int token_padding,
                      int32_t capacity, int B, int32_t NvS,
                      int32_t* z /* R*R */, int32_t* alloc /* R*E */, int32_t* alloc_cumsum /* E*R */,
                      int32_t* experts_to_copy /* R*B */, int32_t* remote_stats /* R*2 */,
                      int32_t* rank_cu_seqlens /* R*(E+B) */, int32_t* rank_zero_fill /* R*(E+B)*2 */,
                      int32_t* expert_offsets /* R*E */, int32_t* dst /* N*K */)
{
    if (N < 0 || E < 1 || K < 1 || R < 1 || E % R != 0 || token_padding < 1 || B < 0 || NvS < 1)
        return ORC_EINVAL;
    const int epn = E / R;
    const int64_t NK = (int64_t)N * K;
    for (int64_t f = 0; f < NK; ++f)
        if (topk[f] < 0 || topk[f] >= E)
            return ORC_EINVAL;

    int32_t* count = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NK > 0 ? NK : 1));
    int32_t* balance = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
    int32_t* quotas = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
    int32_t* remaining = (int32_t*)malloc(sizeof(int32_t) * (size_t)epn);
    int32_t* remote = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    unsigned char* picked = (unsigned char*)malloc((size_t)E);
    unsigned char* seen = (unsigned char*)malloc((size_t)R);
    if (!count || !pos || !balance || !quotas || !remaining || !remote || !picked || !seen) {
        free(count); free(pos); free(balance); free(quotas); free(remaining); free(remote);
        free(picked); free(seen);
        return ORC_ECAP;
    }
    int rc = ORC_OK;

    /* histogram and stable positions */
    for (int64_t f = 0; f < NK; ++f) {
        pos[f] = count[topk[f]];
        count[topk[f]] += 1;
    }

    /* S1 + balance */
    for (int i = 0; i < R * R; ++i)
        z[i] = 0;
    for (int r = 0; r < R; ++r) {
        int32_t g = 0;
        for (int e = r * epn; e < (r + 1) * epn; ++e)
            g += count[e];
        balance[r] = g - capacity;
    }
    for (;;) {
        int s = argmax_low_i32(balance, R);
        int d = argmin_low_i32(balance, R);
        if (balance[s] <= 0 || balance[d] >= 0)
            break;
        int32_t move = -balance[d];
        balance[s] -= move;
        balance[d] = 0;
        z[s * R + d] = move;
    }

    /* alloc per owner rank */
    for (int i = 0; i < R * E; ++i)
        alloc[i] = 0;
    for (int o = 0; o < R; ++o) {
        for (int r = 0; r < R; ++r)
            quotas[r] = z[o * R + r];
        for (int le = 0; le < epn; ++le) {
            remaining[le] = count[o * epn + le];
            alloc[o * E + o * epn + le] = count[o * epn + le];
        }
        for (;;) {
            int t = argmax_low_i32(quotas, R);
            if (quotas[t] <= 0)
                break;
            int le = argmax_low_i32(remaining, epn);
            if (remaining[le] <= 0)
                break;
            int32_t take = remaining[le] < quotas[t] ? remaining[le] : quotas[t];
            quotas[t] -= take;
            remaining[le] -= take;
            alloc[t * E + o * epn + le] += take;
            alloc[o * E + o * epn + le] = remaining[le];
        }
    }
    for (int e = 0; e < E; ++e) {
        int32_t cum = 0;
        for (int r = 0; r < R; ++r) {
            cum += alloc[r * E + e];
            alloc_cumsum[e * R + r] = cum;
        }
    }

    /* selection of redundant experts, per-rank groups */
    for (int i = 0; i < R * 2; ++i)
        remote_stats[i] = 0;
    for (int i = 0; i < R * E; ++i)
        expert_offsets[i] = 0;
    for (int d = 0; d < R && rc == ORC_OK; ++d) {
        int nremote = 0;
        for (int e = 0; e < E; ++e) {
            int local = e >= d * epn && e < (d + 1) * epn;
            remote[e] = local ? 0 : alloc[d * E + e];
            picked[e] = 0;
            if (remote[e] > 0)
                nremote += 1;
        }
        remote_stats[2 * d] = nremote;
        for (int slot = 0; slot < B; ++slot) {
            int best = 0;
            for (int e = 1; e < E; ++e)
                if (remote[e] >= remote[best])
                    best = e; /* ties to the higher index */
            int32_t cnt = remote[best];
            remote[best] = 0;
            int pick = cnt > 0 ? best : -1;
            experts_to_copy[d * B + slot] = pick;
            if (pick >= 0) {
                remote_stats[2 * (pick / epn) + 1] += 1;
                picked[pick] = 1;
            }
        }
        int64_t base = 0;
        for (int g = 0; g < E + B; ++g) {
            int32_t c = 0;
            int expert = -1;
            if (g < E) {
                if (!picked[g]) {
                    c = alloc[d * E + g];
                    expert = g;
                }
            } else {
                int sel = experts_to_copy[d * B + (g - E)];
                if (sel >= 0) {
                    c = alloc[d * E + sel];
                    expert = sel;
                }
            }
            int64_t padded = c > 0 ? ((int64_t)c + token_padding - 1) / token_padding * token_padding : 0;
            if (c > 0)
                expert_offsets[d * E + expert] = (int32_t)base;
            rank_cu_seqlens[d * (E + B) + g] = (int32_t)(base + padded);
            if (c > 0 && padded > c) {
                rank_zero_fill[2 * (d * (E + B) + g)] = (int32_t)(base + c);
                rank_zero_fill[2 * (d * (E + B) + g) + 1] = (int32_t)(padded - c);
            } else {
                rank_zero_fill[2 * (d * (E + B) + g)] = 0;
                rank_zero_fill[2 * (d * (E + B) + g) + 1] = 0;
            }
            base += padded;
        }
        if (base > NvS)
            rc = ORC_ECAP;
    }

    /* dst by the prefix of allocations, then duplicates by rank */
    for (int64_t f = 0; f < NK && rc == ORC_OK; ++f) {
        int e = topk[f];
        int32_t gr = pos[f];
        int r = 0;
        while (alloc_cumsum[e * R + r] <= gr)
            r += 1;
        int32_t pc = r > 0 ? alloc_cumsum[e * R + r - 1] : 0;
        dst[f] = r * NvS + expert_offsets[r * E + e] + (gr - pc);
    }
    for (int s = 0; s < N && rc == ORC_OK; ++s) {
        for (int r = 0; r < R; ++r)
            seen[r] = 0;
        for (int k = 0; k < K; ++k) {
            int64_t f = (int64_t)s * K + k;
            int r = dst[f] / NvS;
            if (seen[r])
                dst[f] = -dst[f] - 1;
            seen[r] = 1;
        }
    }

    free(count); free(pos); free(balance); free(quotas); free(remaining); free(remote);
    free(picked); free(seen);
    return rc;
}

/* ------------------------------------------------------------------ */
/* Grouped-GEMM tile map                                               */
/* ------------------------------------------------------------------ */
/*
 * TensorRT-LLM RoutingKernel.cuh, routingPermutation: for each expert
 * numCta = ceil(count / tile) tiles of `tile` rows; ctaOffset = exclusive
 * prefix of numCta over experts; tile ctaOffset + j (j < numCta) belongs to
 * the expert (CtaIdxXyToBatchIdx) and ends at row
 * min((ctaOffset + j + 1) * tile, ctaOffset * tile + count)
 * (CtaIdxXyToMnLimit); NumNonExitingCtas = sum numCta; PermutedIdxSize =
 * NumNonExitingCtas * tile.  Reading: global expert ids over all experts
 * (the page filters a rank's local experts), and tiles from num_tiles up to
 * max_tiles hold -1.
 */
int orc_tile_map(const int32_t* counts, int E, int tile, int32_t* tile_expert, int32_t* tile_row_limit,
                 int64_t max_tiles, int32_t* sizes)
{
    if (E < 1 || tile < 1)
        return ORC_EINVAL;
    int64_t cta_offset = 0;
    for (int e = 0; e < E; ++e) {
        if (counts[e] < 0)
            return ORC_EINVAL;
        int64_t num_cta = ((int64_t)counts[e] + tile - 1) / tile;
        for (int64_t j = 0; j < num_cta; ++j) {
            int64_t t = cta_offset + j;
            if (t >= max_tiles)
                return ORC_ECAP;
            int64_t lim1 = (cta_offset + j + 1) * tile;
            int64_t lim2 = cta_offset * tile + counts[e];
            tile_expert[t] = e;
            tile_row_limit[t] = (int32_t)(lim1 < lim2 ? lim1 : lim2);
        }
        cta_offset += num_cta;
    }
    for (int64_t t = cta_offset; t < max_tiles; ++t) {
        tile_expert[t] = -1;
        tile_row_limit[t] = -1;
    }
    sizes[0] = (int32_t)cta_offset;
    sizes[1] = (int32_t)(cta_offset * tile);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Rank layout: channel prefix matrix, deduplicated per-rank slots      */
/* ------------------------------------------------------------------ */
/*
 * DeepEP csrc/kernels/intranode.cu, notify_dispatch: for each destination
 * rank and channel, the number of the channel's tokens that go to the rank
 * (is_token_in_rank), then an inclusive prefix over channels
 * (channel_prefix_matrix[r][c]).  Reading: channel c covers tokens
 * [min(c*q, N), min((c+1)*q, N)) with q = ceil(N / C) (the helper that
 * splits tokens is not on the page).
 * token_rank_slot[s][r]: reading of DeepEP's per-(token, rank) send slot
 * with one source rank: a token goes to each rank it needs exactly once,
 * ranks' blocks follow each other (rank_prefix = exclusive prefix of
 * tokens per rank) and tokens keep their order inside a block:
 * rank_prefix[r] + #{s' < s : is_token_in_rank[s'][r]}, or -1.
 */
int orc_rank_layout(const uint8_t* is_token_in_rank, int N, int R, int C, int32_t* channel_prefix_matrix,
                    int32_t* token_rank_slot)
{
    if (N < 0 || R < 1 || C < 1)
        return ORC_EINVAL;
    int64_t q = ((int64_t)N + C - 1) / C;
    int32_t base = 0;
    for (int r = 0; r < R; ++r) {
        int32_t run = 0;
        for (int c = 0; c < C; ++c) {
            int64_t b = (int64_t)c * q < N ? (int64_t)c * q : N;
            int64_t e = ((int64_t)c + 1) * q < N ? ((int64_t)c + 1) * q : N;
            for (int64_t s = b; s < e; ++s)
                run += is_token_in_rank[s * R + r] ? 1 : 0;
            channel_prefix_matrix[r * C + c] = run;
        }
        int32_t pos = 0;
        for (int64_t s = 0; s < N; ++s) {
            if (is_token_in_rank[s * R + r]) {
                token_rank_slot[s * R + r] = base + pos;
                pos += 1;
            } else {
                token_rank_slot[s * R + r] = -1;
            }
        }
        base += pos;
    }
    return ORC_OK;
}
