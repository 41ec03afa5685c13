// route_core.cuh -- the router's arithmetic for one GPU (sm_103a), shared by
// the routing kernel and the fused route + plan kernel.
//
// A group of G lanes (G = 2..32) owns one token.  Each lane holds its share
// of the fp32 logit row, forms the selection key in registers, and K rounds
// of a warp arg-max pick the experts: the largest key wins, equal keys go to
// the lower expert index (MoonEP moonep/planning.py, warp_argmax_min_idx: a
// max reduction on the value, then a min reduction on the index among lanes
// holding that value).  With G = 32 the two reductions are single
// redux.sync instructions; with smaller groups an xor butterfly over (key,
// index, value) does the same.
//
// Scores (TensorRT-LLM RoutingKernel.cuh, calcSoftmax / sigmoid_accurate):
//   softmax: the key is the logit itself (softmax is increasing), weights
//            are the softmax over the K selected logits (or over the row);
//   sigmoid: key = sigmoid(logit) + bias in fp32, the sigmoid evaluated by
//            one fixed operation sequence so that the ordering is
//            reproducible bit for bit (see sigmoid_f32 below).
// Group-limited selection (sigmoid only): the group score is the fp32 sum
// of the group's two largest keys, the topk_group best groups (ties to the
// lower group) stay eligible.
#pragma once

#include "moe_common.cuh"

namespace moe {

// ---------------------------------------------------------------- fp32 exp / sigmoid
__device__ __forceinline__ float pow2_int(int n) { return __int_as_float((n + 127) << 23); }

// e^t for t <= 0.  Cody & Waite argument reduction t = n ln2 + r with
// |r| <= ln2/2 and ln2 split into a 16-significant-bit head (so n*head is
// exact) and an fp32 tail; e^r by its degree-7 Taylor polynomial (1/j!)
// in Horner form, one fused multiply-add per step; then 2^n applied as two
// exact power-of-two factors so intermediate results stay normal.
// No branches (lanes of a warp take the same path whatever their t): out of
// range inputs are clamped for the arithmetic and replaced at the end.
__device__ __forceinline__ float exp_nonpos(float t_in) {
    const float t = fmaxf(fminf(t_in, 0.0f), -105.0f);      // NaN -> -105, fixed below
    const float nf = rintf(__fmul_rn(t, 0x1.715476p+0f));  // t / ln2
    float r = __fmaf_rn(-nf, 0x1.62e4p-1f, t);              // - n * ln2 (head)
    r = __fmaf_rn(-nf, 0x1.7f7d1cp-20f, r);                 // - n * ln2 (tail)
    float p = 0x1.a01a02p-13f;                              // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);                   // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);                    // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);                    // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);                    // 1/3!
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int n = static_cast<int>(nf);  // -152 <= n <= 0, exact
    const int n1 = n / 2;
    const int n2 = n - n1;
    const float e = __fmul_rn(__fmul_rn(p, pow2_int(n1)), pow2_int(n2));
    return t_in != t_in ? t_in : (t_in < -104.0f ? 0.0f : e);
}

// sigmoid(x) = 1 / (1 + e^-x) for x >= 0 and e^x / (1 + e^x) below, each
// operation rounded once (IEEE division, no flush of subnormals).
// One path for both signs (numerator selected), so a warp evaluates one
// exponential and one division per value.
__device__ __forceinline__ float sigmoid_f32(float x) {
    const bool pos = x >= 0.0f;
    const float e = exp_nonpos(pos ? -x : x);
    const float q = __fdiv_rn(pos ? 1.0f : e, __fadd_rn(1.0f, e));
    return x != x ? x : q;
}

// Monotone map fp32 -> uint32 (larger float -> larger integer); -0 is
// folded onto +0 so the two compare equal as floats do.  0 sits below every
// non-NaN value and marks used or ineligible experts.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(__fadd_rn(f, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// e^(a - b) for a <= b, with the rounding error of the subtraction carried
// to first order (TwoSum), so only the exponential's own error remains.
__device__ __forceinline__ float exp_diff(float a, float b) {
    const float s = __fsub_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(-b, bb));
    const float e = exp_nonpos(s);
    return __fmaf_rn(e, err, e);
}

// Float-float accumulation (hi + lo, |lo| <= ulp(hi)/2) of non-negative
// terms: TwoSum of the heads, tails added, Fast2Sum renormalisation.
__device__ __forceinline__ void ff_add(float& hi, float& lo, float bh, float bl) {
    const float s = __fadd_rn(hi, bh);
    const float bb = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(bh, bb));
    const float t = __fadd_rn(__fadd_rn(lo, bl), err);
    hi = __fadd_rn(s, t);
    lo = __fsub_rn(t, __fsub_rn(hi, s));
}

// A winner's score for its weight: the same 1/(1+e^-x) (x >= 0) or
// e^x/(1+e^x) as the key, with the rounding error of 1+e carried to first
// order, so only e's own error (about 1 ulp) and two roundings remain.
__device__ __forceinline__ float sigmoid_weight(float x) {
    const bool pos = x >= 0.0f;
    const float e = exp_nonpos(pos ? -x : x);
    const float d = __fadd_rn(1.0f, e);
    const float dlo = __fsub_rn(e, __fsub_rn(d, 1.0f));  // exact: 1 + e = d + dlo
    const float q = __fdiv_rn(pos ? 1.0f : e, d);
    return __fmaf_rn(-q, __fdiv_rn(dlo, d), q);
}

// A lane's two largest keys not yet taken, with their slots and values.
// Strict comparisons: equal keys keep the lower slot (slots ascend in
// expert index), as the arg-max tie rule wants.
template <int V>
__device__ __forceinline__ void lane_top2(const uint32_t (&key)[V], const float (&raw)[V], uint32_t taken,
                                          uint32_t& k1, int& j1, float& v1, uint32_t& k2, int& j2, float& v2) {
    k1 = 0u;
    k2 = 0u;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const uint32_t kv = ((taken >> v) & 1u) ? 0u : key[v];
        if (kv > k1) {
            k2 = k1;
            j2 = j1;
            v2 = v1;
            k1 = kv;
            j1 = v;
            v1 = raw[v];
        } else if (kv > k2) {
            k2 = kv;
            j2 = v;
            v2 = raw[v];
        }
    }
}

struct RouteArgs {
    const float* logits;
    const float* bias;
    int32_t* topk_idx;
    float* topk_w;
    int N, E, K, scoring, renormalize, n_group, topk_group;
    float scaling;
};

constexpr int ROUTE_THREADS = 128;

// G lanes per token; V values per lane; VEC: values come as float4 at
// experts 4*(sub + G*j) + q, otherwise one value at sub + G*v.
template <int G, int V, bool VEC>
__device__ __forceinline__ int expert_of(int sub, int v) {
    if constexpr (VEC) {
        return 4 * (sub + G * (v / 4)) + (v % 4);
    } else {
        return sub + G * v;
    }
}

template <int G, int V, bool VEC>
__device__ __forceinline__ void load_row(const RouteArgs& a, int64_t s, int sub, float (&raw)[V]) {
    const bool valid = s < a.N;
    const float* row = a.logits + (valid ? s : 0) * a.E;
    if constexpr (VEC) {
#pragma unroll
        for (int j = 0; j < V / 4; ++j) {
            const int e0 = 4 * (sub + G * j);
            float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
            if (valid && e0 < a.E) q = ld_stream_f4(row + e0);
            raw[4 * j + 0] = q.x;
            raw[4 * j + 1] = q.y;
            raw[4 * j + 2] = q.z;
            raw[4 * j + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int e = sub + G * v;
            raw[v] = (valid && e < a.E) ? ld_stream_f32(row + e) : 0.f;
        }
    }
}

// Route one token: its G lanes call this together (lane `sub` of the group,
// `lane` its lane in the warp), each with the logits of its experts as
// expert_of lays them out (raw) and their bias (bias_r).  Lane `sub` gets
// the winners k = sub, sub + G, ...: my_idx[t], num[t] for k = sub + G t < K.
// s_keys: the warp's row of E floats (general group-limited path only).
template <int G, int V, bool VEC, int KMAX>
__device__ __forceinline__ void route_token(const RouteArgs& a, const float (&raw)[V], const float (&bias_r)[V],
                                            bool valid, int lane, int sub, float* s_keys,
                                            int (&my_idx)[(KMAX + G - 1) / G], float (&num)[(KMAX + G - 1) / G]) {
    constexpr int KPL = (KMAX + G - 1) / G;  // winners kept per lane
    const int E = a.E, K = a.K;
    const bool sigmoid = a.scoring == MOE_SCORING_SIGMOID;
    const bool grouped = a.n_group > 1;
    const bool has_bias = a.bias != nullptr;
    const int gs = E / a.n_group;
    // Register path for group scores: a group is a run of L = gs/4 lanes
    // of one float4 slot (needs G = 32, float4 rows, L a power of two).
    const int L = gs / 4;
    const bool gfast = G == 32 && VEC && grouped && gs % 4 == 0 && L >= 1 && L <= 32 && (L & (L - 1)) == 0;

    // ---- keys
    float keyf[V];
    uint32_t key[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int e = expert_of<G, V, VEC>(sub, v);
        if (sigmoid) {
            const float sg = sigmoid_f32(raw[v]);
            keyf[v] = has_bias ? __fadd_rn(sg, bias_r[v]) : sg;
        } else {
            keyf[v] = raw[v];
        }
        key[v] = (valid && e < E) ? order_key(keyf[v]) : 0u;
    }

    // ---- group-limited eligibility
    if constexpr (G == 32) {
        if (grouped) {
            uint32_t kept = 0u;
            if (gfast) {
                // top-2 of each lane's float4, merged over the group's lanes
                float sc[V / 4 > 0 ? V / 4 : 1];
#pragma unroll
                for (int j = 0; j < V / 4; ++j) {
                    const float x0 = keyf[4 * j], x1 = keyf[4 * j + 1], x2 = keyf[4 * j + 2], x3 = keyf[4 * j + 3];
                    const float hi01 = fmaxf(x0, x1), lo01 = fminf(x0, x1);
                    const float hi23 = fmaxf(x2, x3), lo23 = fminf(x2, x3);
                    float m1 = fmaxf(hi01, hi23);
                    float m2 = fmaxf(fminf(hi01, hi23), fmaxf(lo01, lo23));
                    for (int off = 1; off < L; off <<= 1) {
                        const float o1 = __shfl_xor_sync(FULL_MASK, m1, off);
                        const float o2 = __shfl_xor_sync(FULL_MASK, m2, off);
                        const float n1 = fmaxf(m1, o1);
                        m2 = fmaxf(fminf(m1, o1), fmaxf(m2, o2));
                        m1 = n1;
                    }
                    sc[j] = __fadd_rn(m1, m2);
                }
                const int lsh = __ffs(L) - 1;        // L is a power of two
                const int gpj = 32 >> lsh;           // groups per float4 slot
                const int lgrp = lane >> lsh;        // this lane's group within a slot
                const bool lead = (lane & (L - 1)) == 0;
                uint32_t taken = 0u;     // candidate slots of this lane already kept
                for (int r = 0; r < a.topk_group; ++r) {
                    uint32_t ck = 0u, cg = 32u;
#pragma unroll
                    for (int j = 0; j < V / 4; ++j) {
                        const int g = j * gpj + lgrp;
                        const bool cand = lead && g < a.n_group && !((taken >> j) & 1u);
                        const uint32_t k2 = cand ? order_key(sc[j]) : 0u;
                        if (k2 > ck) {
                            ck = k2;
                            cg = static_cast<uint32_t>(g);
                        }
                    }
                    const uint32_t m = __reduce_max_sync(FULL_MASK, ck);
                    const uint32_t win = __reduce_min_sync(FULL_MASK, ck == m ? cg : 32u);
                    kept |= 1u << win;
#pragma unroll
                    for (int j = 0; j < V / 4; ++j)
                        if (lead && static_cast<uint32_t>(j * gpj + lgrp) == win) taken |= 1u << j;
                }
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int g = (v / 4) * gpj + lgrp;
                    if (!((kept >> g) & 1u)) key[v] = 0u;
                }
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int e = expert_of<G, V, VEC>(sub, v);
                    if (e < E) s_keys[e] = keyf[v];
                }
                __syncwarp();
                uint32_t gkey = 0u;
                if (lane < a.n_group) {
                    float m1 = -INFINITY, m2 = -INFINITY;
                    for (int j = 0; j < gs; ++j) {
                        const float x = s_keys[lane * gs + j];
                        if (x > m1) {
                            m2 = m1;
                            m1 = x;
                        } else if (x > m2) {
                            m2 = x;
                        }
                    }
                    gkey = order_key(gs == 1 ? m1 : __fadd_rn(m1, m2));
                }
                for (int r = 0; r < a.topk_group; ++r) {
                    const uint32_t m = __reduce_max_sync(FULL_MASK, gkey);
                    const uint32_t win =
                        __reduce_min_sync(FULL_MASK, gkey == m ? static_cast<uint32_t>(lane) : 32u);
                    kept |= 1u << win;
                    if (static_cast<uint32_t>(lane) == win) gkey = 0u;
                }
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int e = expert_of<G, V, VEC>(sub, v);
                    if (e < E && !((kept >> (e / gs)) & 1u)) key[v] = 0u;
                }
                __syncwarp();
            }
        }
    }

    // ---- K rounds of arg-max
    float my_val[KPL];
    float top_val = 0.f;
    if constexpr (G == 32) {
        // each lane caches its two best (key, slot, value); a lane whose
        // cache runs dry rescans its keys minus the ones already taken,
        // only when it still has some and only then (rare with K <= 8)
        uint32_t k1 = 0u, k2 = 0u, taken = 0u;
        int j1 = 0, j2 = 0;
        float v1 = 0.f, v2 = 0.f;
        lane_top2<V>(key, raw, taken, k1, j1, v1, k2, j2, v2);
        int left = 0;  // this lane's eligible keys not yet taken
#pragma unroll
        for (int v = 0; v < V; ++v) left += key[v] != 0u ? 1 : 0;
        bool dry = false;
#pragma unroll
        for (int r = 0; r < KMAX; ++r) {
            if (r >= K) break;
            if (__any_sync(FULL_MASK, dry)) {
                if (dry) lane_top2<V>(key, raw, taken, k1, j1, v1, k2, j2, v2);
                dry = false;
            }
            const uint32_t i1 = k1 != 0u ? static_cast<uint32_t>(expert_of<G, V, VEC>(sub, j1)) : 0xffffffffu;
            const uint32_t m = __reduce_max_sync(FULL_MASK, k1);
            const uint32_t wi = __reduce_min_sync(FULL_MASK, k1 == m ? i1 : 0xffffffffu);
            const int owner = VEC ? static_cast<int>((wi / 4) % G) : static_cast<int>(wi % G);
            const float wv = __shfl_sync(FULL_MASK, v1, owner);
            if (i1 == wi) {  // this lane's best won: pop it
                taken |= 1u << j1;
                --left;
                k1 = k2;
                j1 = j2;
                v1 = v2;
                k2 = 0u;
                dry = k1 == 0u && left > 0;
            }
            if (r == 0) top_val = wv;
            if (r == sub) {
                my_idx[0] = static_cast<int>(wi);
                my_val[0] = wv;
            }
        }
    } else {
        // each lane keeps its best and rescans only when its best wins
        uint32_t bk = 0u, bi = 0xffffffffu;
        float bv = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v)
            if (key[v] > bk) {  // values ascend in expert index per lane
                bk = key[v];
                bi = static_cast<uint32_t>(expert_of<G, V, VEC>(sub, v));
                bv = raw[v];
            }
#pragma unroll
        for (int r = 0; r < KMAX; ++r) {
            if (r >= K) break;
            uint32_t ck = bk, ci = bi;
            float cv = bv;
#pragma unroll
            for (int off = 1; off < G; off <<= 1) {
                const uint32_t ok = __shfl_xor_sync(FULL_MASK, ck, off);
                const uint32_t oi = __shfl_xor_sync(FULL_MASK, ci, off);
                const float ov = __shfl_xor_sync(FULL_MASK, cv, off);
                if (ok > ck || (ok == ck && oi < ci)) {
                    ck = ok;
                    ci = oi;
                    cv = ov;
                }
            }
            const uint32_t wi = ci;
            const float wv = cv;
            if (bi == wi) {  // this lane owned the winner: drop it, find its next best
#pragma unroll
                for (int v = 0; v < V; ++v)
                    if (static_cast<uint32_t>(expert_of<G, V, VEC>(sub, v)) == wi) key[v] = 0u;
                bk = 0u;
                bi = 0xffffffffu;
#pragma unroll
                for (int v = 0; v < V; ++v)
                    if (key[v] > bk) {
                        bk = key[v];
                        bi = static_cast<uint32_t>(expert_of<G, V, VEC>(sub, v));
                        bv = raw[v];
                    }
            }
            if (r == 0) top_val = wv;
            if (r % G == sub) {
                my_idx[r / G] = static_cast<int>(wi);
                my_val[r / G] = wv;
            }
        }
    }

    // ---- weights: lane `sub` owns winners k = sub, sub + G, ...
    float shi = 0.f, slo = 0.f;  // this lane's part of the normaliser
#pragma unroll
    for (int t = 0; t < KPL; ++t) {
        const int k = sub + G * t;
        num[t] = 0.f;
        if (k >= K) continue;
        if (!sigmoid) {
            num[t] = exp_diff(my_val[t], top_val);  // top-1 logit is the row maximum
        } else {
            num[t] = sigmoid_weight(my_val[t]);
        }
        if (a.renormalize && (!sigmoid || num[t] >= 0x1p-100f)) ff_add(shi, slo, num[t], 0.f);
    }
    if (!sigmoid && !a.renormalize) {  // full-row softmax normaliser
        shi = 0.f;
        slo = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int e = expert_of<G, V, VEC>(sub, v);
            if (valid && e < E) ff_add(shi, slo, exp_diff(raw[v], top_val), 0.f);
        }
    }
    bool tiny = false;  // a sigmoid score below 2^-100: fp64 for this token
    if (sigmoid) {
#pragma unroll
        for (int t = 0; t < KPL; ++t)
            if (sub + G * t < K && num[t] < 0x1p-100f) tiny = true;
    }
    if (__any_sync(FULL_MASK, tiny)) {
        // rare: recompute the warp's scores and normalisers in fp64
        // (the reduction stays inside each token's group of G lanes)
        double sd[KPL], den = 0.0;
#pragma unroll
        for (int t = 0; t < KPL; ++t) {
            const int k = sub + G * t;
            sd[t] = 0.0;
            if (k < K) {
                const double ex = exp(-fabs(static_cast<double>(my_val[t])));
                sd[t] = my_val[t] >= 0.f ? 1.0 / (1.0 + ex) : ex / (1.0 + ex);
            }
            den += sd[t];
        }
#pragma unroll
        for (int off = 1; off < G; off <<= 1) den += __shfl_xor_sync(FULL_MASK, den, off);
        const double scale = a.renormalize ? static_cast<double>(a.scaling) / den : a.scaling;
#pragma unroll
        for (int t = 0; t < KPL; ++t) num[t] = static_cast<float>(sd[t] * scale);
    } else {
#pragma unroll
        for (int off = 1; off < G; off <<= 1) {
            const float oh = __shfl_xor_sync(FULL_MASK, shi, off);
            const float ol = __shfl_xor_sync(FULL_MASK, slo, off);
            ff_add(shi, slo, oh, ol);
        }
        if (a.renormalize || !sigmoid) {
            // w = num * scaling / (shi + slo): one correctly rounded
            // division, then the tail of the normaliser to first order
            const float q = __fdiv_rn(a.scaling, shi);
            const float qc = __fmaf_rn(-q, __fdiv_rn(slo, shi), q);
#pragma unroll
            for (int t = 0; t < KPL; ++t) num[t] = __fmul_rn(num[t], qc);
        } else {
#pragma unroll
            for (int t = 0; t < KPL; ++t) num[t] = __fmul_rn(num[t], a.scaling);
        }
    }

}

// The bias of a lane's experts (zero without bias or for softmax scores).
template <int G, int V, bool VEC>
__device__ __forceinline__ void lane_bias(const RouteArgs& a, int sub, float (&bias_r)[V]) {
    const bool sigmoid = a.scoring == MOE_SCORING_SIGMOID;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int e = expert_of<G, V, VEC>(sub, v);
        bias_r[v] = (sigmoid && a.bias != nullptr && e < a.E) ? __ldg(a.bias + e) : 0.0f;
    }
}

}  // namespace moe

namespace moe_host {

// Host checks of a routing call and its argument block (shared by
// moe_route_topk and the fused moe_route_plan): MOE_OK or the error code.
inline int route_args(const float* logits, const float* bias, int N, int E, int K, int scoring, int renormalize,
                      int n_group, int topk_group, float routed_scaling, int32_t* topk_idx, float* topk_w,
                      moe::RouteArgs* a) {
    auto aligned = [](const void* p, uintptr_t al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; };
    // N = 0 (an empty batch) is valid; its zero-sized arrays may be null
    if (N > 0 && (logits == nullptr || topk_idx == nullptr || topk_w == nullptr)) return MOE_ERR_INVALID_ARG;
    if (N < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOE_ERR_INVALID_ARG;
    if (scoring != MOE_SCORING_SOFTMAX && scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (n_group < 1 || n_group > 32) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(N) * K >= (int64_t(1) << 31) || static_cast<int64_t>(N) * E >= (int64_t(1) << 40))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4)) return MOE_ERR_INVALID_ARG;
    if (E % 4 == 0 && !aligned(logits, 16)) return MOE_ERR_INVALID_ARG;
    if (bias != nullptr && (scoring != MOE_SCORING_SIGMOID || !aligned(bias, 4))) return MOE_ERR_UNSUPPORTED;
    if (n_group > 1) {
        if (scoring != MOE_SCORING_SIGMOID) return MOE_ERR_UNSUPPORTED;
        if (E % n_group != 0 || topk_group < 1 || topk_group > n_group || K > topk_group * (E / n_group))
            return MOE_ERR_INVALID_ARG;
    }
    if (!(routed_scaling == routed_scaling)) return MOE_ERR_INVALID_ARG;
    a->logits = logits;
    a->bias = bias;
    a->topk_idx = topk_idx;
    a->topk_w = topk_w;
    a->N = N;
    a->E = E;
    a->K = K;
    a->scoring = scoring;
    a->renormalize = renormalize ? 1 : 0;
    a->n_group = n_group;
    a->topk_group = n_group > 1 ? topk_group : 1;
    a->scaling = routed_scaling;
    return MOE_OK;
}

}  // namespace moe_host
