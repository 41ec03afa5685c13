// route.cu -- router top-K for one GPU (sm_103a).
//
// A group of G lanes (G = 2..32) owns one token.  Each lane streams its
// share of the fp32 logit row with 16-byte non-allocating loads, forms the
// selection key in registers, and K rounds of a warp arg-max pick the
// experts: the largest key wins, equal keys go to the lower expert index
// (MoonEP moonep/planning.py, warp_argmax_min_idx: a max reduction on the
// value, then a min reduction on the index among lanes holding that value).
// With G = 32 the two reductions are single redux.sync instructions; with
// smaller groups an xor butterfly over (key, index, value) does the same.
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
#include "moe_common.cuh"

namespace moe {

// ---------------------------------------------------------------- fp32 exp / sigmoid
__device__ __forceinline__ float pow2_int(int n) { return __int_as_float((n + 127) << 23); }

// e^t for t <= 0.  Cody & Waite argument reduction t = n ln2 + r with
// |r| <= ln2/2 and ln2 split into a 16-significant-bit head (so n*head is
// exact) and an fp32 tail; e^r by its degree-7 Taylor polynomial (1/j!)
// in Horner form, one fused multiply-add per step; then 2^n applied as two
// exact power-of-two factors so intermediate results stay normal.
__device__ __forceinline__ float exp_nonpos(float t) {
    if (t != t) return t;
    if (t > 0.0f) t = 0.0f;
    if (t < -104.0f) return 0.0f;
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
    const int n = static_cast<int>(nf);  // -150 <= n <= 0, exact
    const int n1 = n / 2;
    const int n2 = n - n1;
    return __fmul_rn(__fmul_rn(p, pow2_int(n1)), pow2_int(n2));
}

// sigmoid(x) = 1 / (1 + e^-x) for x >= 0 and e^x / (1 + e^x) below, each
// operation rounded once (IEEE division, no flush of subnormals).
__device__ __forceinline__ float sigmoid_f32(float x) {
    if (x != x) return x;
    if (x >= 0.0f) {
        const float e = exp_nonpos(-x);
        return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
    }
    const float e = exp_nonpos(x);
    return __fdiv_rn(e, __fadd_rn(1.0f, e));
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

template <int G, int V, bool VEC, int KMAX>
__global__ void __launch_bounds__(ROUTE_THREADS) route_topk_kernel(const RouteArgs a) {
    extern __shared__ float s_keys_all[];  // [warps][E], group-limited only
    pdl_wait();
    pdl_trigger();

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane % G;
    const int group_base = lane - sub;
    constexpr int TPW = 32 / G;  // tokens per warp
    const int E = a.E, K = a.K;
    const bool sigmoid = a.scoring == MOE_SCORING_SIGMOID;
    float* s_keys = s_keys_all + warp * E;

    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (ROUTE_THREADS / 32);
    for (int64_t wtok = (static_cast<int64_t>(blockIdx.x) * (ROUTE_THREADS / 32) + warp) * TPW;
         wtok < a.N; wtok += warps_total * TPW) {
        const int64_t s = wtok + lane / G;
        const bool valid = s < a.N;
        const float* row = a.logits + (valid ? s : 0) * E;

        // ---- load and score
        float raw[V];  // logits
        float keyf[V];
        if constexpr (VEC) {
#pragma unroll
            for (int j = 0; j < V / 4; ++j) {
                const int e0 = 4 * (sub + G * j);
                float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
                if (valid && e0 < E) q = ld_stream_f4(row + e0);
                raw[4 * j + 0] = q.x;
                raw[4 * j + 1] = q.y;
                raw[4 * j + 2] = q.z;
                raw[4 * j + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int e = sub + G * v;
                raw[v] = (valid && e < E) ? ld_stream_f32(row + e) : 0.f;
            }
        }
        uint32_t key[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int e = expert_of<G, V, VEC>(sub, v);
            if (sigmoid) {
                const float sg = sigmoid_f32(raw[v]);
                keyf[v] = a.bias != nullptr && e < E ? __fadd_rn(sg, __ldg(a.bias + e)) : sg;
            } else {
                keyf[v] = raw[v];
            }
            key[v] = (valid && e < E) ? order_key(keyf[v]) : 0u;
        }

        // ---- group-limited eligibility (G == 32 only; host enforces)
        if constexpr (G == 32) {
            if (a.n_group > 1) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int e = expert_of<G, V, VEC>(sub, v);
                    if (e < E) s_keys[e] = keyf[v];
                }
                __syncwarp();
                const int gs = E / a.n_group;
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
                uint32_t kept = 0u;
                for (int r = 0; r < a.topk_group; ++r) {
                    const uint32_t m = __reduce_max_sync(FULL_MASK, gkey);
                    const uint32_t win = __reduce_min_sync(FULL_MASK, gkey == m ? static_cast<uint32_t>(lane) : 32u);
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

        // ---- K rounds of arg-max
        int win_idx[KMAX];
        float win_val[KMAX];
#pragma unroll
        for (int r = 0; r < KMAX; ++r) {
            if (r >= K) break;
            uint32_t bk = 0u, bi = 0xffffffffu;
            float bv = 0.f;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if (key[v] > bk) {  // values ascend in expert index per lane
                    bk = key[v];
                    bi = static_cast<uint32_t>(expert_of<G, V, VEC>(sub, v));
                    bv = raw[v];
                }
            }
            uint32_t wi;
            float wv;
            if constexpr (G == 32) {
                const uint32_t m = __reduce_max_sync(FULL_MASK, bk);
                wi = __reduce_min_sync(FULL_MASK, bk == m ? bi : 0xffffffffu);
                const int owner = VEC ? static_cast<int>((wi / 4) % G) : static_cast<int>(wi % G);
                wv = __shfl_sync(FULL_MASK, bv, owner);
            } else {
#pragma unroll
                for (int off = 1; off < G; off <<= 1) {
                    const uint32_t ok = __shfl_xor_sync(FULL_MASK, bk, off);
                    const uint32_t oi = __shfl_xor_sync(FULL_MASK, bi, off);
                    const float ov = __shfl_xor_sync(FULL_MASK, bv, off);
                    if (ok > bk || (ok == bk && oi < bi)) {
                        bk = ok;
                        bi = oi;
                        bv = ov;
                    }
                }
                wi = bi;
                wv = bv;
            }
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if (static_cast<uint32_t>(expert_of<G, V, VEC>(sub, v)) == wi) key[v] = 0u;
            }
            win_idx[r] = static_cast<int>(wi);
            win_val[r] = wv;
        }

        // ---- weights (win_val holds the winners' logits)
        float w[KMAX];
        if (!sigmoid) {
            const float m = win_val[0];  // top-1 logit is the row maximum
            float ek[KMAX];
            double denom = 0.0;
#pragma unroll
            for (int r = 0; r < KMAX; ++r) {
                if (r >= K) break;
                ek[r] = exp_diff(win_val[r], m);
                denom += static_cast<double>(ek[r]);
            }
            if (!a.renormalize) {
                double part = 0.0;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int e = expert_of<G, V, VEC>(sub, v);
                    if (valid && e < E) part += static_cast<double>(exp_diff(raw[v], m));
                }
#pragma unroll
                for (int off = 1; off < G; off <<= 1) part += __shfl_xor_sync(FULL_MASK, part, off);
                denom = part;
            }
            const double scale = static_cast<double>(a.scaling) / denom;
#pragma unroll
            for (int r = 0; r < KMAX; ++r) {
                if (r >= K) break;
                w[r] = static_cast<float>(static_cast<double>(ek[r]) * scale);
            }
        } else {
            // scores of the winners; below 2^-100 the fp32 score has lost
            // relative precision (or underflowed), so fp64 takes over there
            double sc[KMAX];
            double denom = 0.0;
#pragma unroll
            for (int r = 0; r < KMAX; ++r) {
                if (r >= K) break;
                const float sf = sigmoid_f32(win_val[r]);
                if (sf < 0x1p-100f) {
                    const double ex = exp(static_cast<double>(win_val[r]));
                    sc[r] = ex / (1.0 + ex);
                } else {
                    sc[r] = static_cast<double>(sf);
                }
                denom += sc[r];
            }
            const double scale = a.renormalize ? static_cast<double>(a.scaling) / denom
                                               : static_cast<double>(a.scaling);
#pragma unroll
            for (int r = 0; r < KMAX; ++r) {
                if (r >= K) break;
                w[r] = static_cast<float>(sc[r] * scale);
            }
        }

        // ---- store: lane `sub` writes k = sub, sub + G, ...
        if (valid) {
#pragma unroll
            for (int r = 0; r < KMAX; ++r) {
                if (r >= K) break;
                if (r % G == sub) {
                    a.topk_idx[s * K + r] = win_idx[r];
                    a.topk_w[s * K + r] = w[r];
                }
            }
        }
        (void)group_base;
    }
}

}  // namespace moe

// ---------------------------------------------------------------- host
namespace {

using moe::RouteArgs;

template <int G, int V, bool VEC, int KMAX>
int launch_route(const RouteArgs& a, cudaStream_t stream) {
    const int tokens_per_block = moe::ROUTE_THREADS / G;
    int64_t blocks = (static_cast<int64_t>(a.N) + tokens_per_block - 1) / tokens_per_block;
    const int64_t cap = static_cast<int64_t>(moe_host::num_sms()) * 16;
    if (blocks > cap) blocks = cap;
    const size_t smem = (a.n_group > 1) ? sizeof(float) * a.E * (moe::ROUTE_THREADS / 32) : 0;
    return moe_host::launch(moe::route_topk_kernel<G, V, VEC, KMAX>, dim3(static_cast<unsigned>(blocks)),
                            dim3(moe::ROUTE_THREADS), smem, stream, a);
}

template <int KMAX>
int dispatch_route(const RouteArgs& a, cudaStream_t stream) {
    const int E = a.E;
    const bool grouped = a.n_group > 1;
    if (E % 4 == 0) {
        if (!grouped && E <= 8) return launch_route<2, 4, true, KMAX>(a, stream);
        if (!grouped && E <= 16) return launch_route<4, 4, true, KMAX>(a, stream);
        if (!grouped && E <= 32) return launch_route<8, 4, true, KMAX>(a, stream);
        if (!grouped && E <= 64) return launch_route<16, 4, true, KMAX>(a, stream);
        if (E <= 128) return launch_route<32, 4, true, KMAX>(a, stream);
        if (E <= 256) return launch_route<32, 8, true, KMAX>(a, stream);
        if (E <= 512) return launch_route<32, 16, true, KMAX>(a, stream);
        return launch_route<32, 32, true, KMAX>(a, stream);
    }
    if (E <= 32) return launch_route<32, 1, false, KMAX>(a, stream);
    if (E <= 64) return launch_route<32, 2, false, KMAX>(a, stream);
    if (E <= 128) return launch_route<32, 4, false, KMAX>(a, stream);
    if (E <= 256) return launch_route<32, 8, false, KMAX>(a, stream);
    if (E <= 512) return launch_route<32, 16, false, KMAX>(a, stream);
    return launch_route<32, 32, false, KMAX>(a, stream);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" MOE_API int moe_route_topk(const float* logits, const float* bias, int N, int E, int K,
                                      int scoring, int renormalize, int n_group, int topk_group,
                                      float routed_scaling, int32_t* topk_idx, float* topk_w,
                                      cudaStream_t stream) {
    if (logits == nullptr || topk_idx == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
    if (N < 1 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOE_ERR_INVALID_ARG;
    if (scoring != MOE_SCORING_SOFTMAX && scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (n_group < 1 || n_group > 32) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(N) * K >= (int64_t(1) << 31) || static_cast<int64_t>(N) * E >= (int64_t(1) << 40))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4)) return MOE_ERR_INVALID_ARG;
    if (E % 4 == 0 && !aligned(logits, 16)) return MOE_ERR_INVALID_ARG;
    if (bias != nullptr && (scoring != MOE_SCORING_SIGMOID || !aligned(bias, 4))) return MOE_ERR_UNSUPPORTED;
    if (n_group > 1) {
        if (scoring != MOE_SCORING_SIGMOID) return MOE_ERR_UNSUPPORTED;
        if (E % n_group != 0 || topk_group < 1 || topk_group > n_group ||
            K > topk_group * (E / n_group))
            return MOE_ERR_INVALID_ARG;
    }
    if (!(routed_scaling == routed_scaling)) return MOE_ERR_INVALID_ARG;

    RouteArgs a;
    a.logits = logits;
    a.bias = bias;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.N = N;
    a.E = E;
    a.K = K;
    a.scoring = scoring;
    a.renormalize = renormalize ? 1 : 0;
    a.n_group = n_group;
    a.topk_group = n_group > 1 ? topk_group : 1;
    a.scaling = routed_scaling;
    return K <= 8 ? dispatch_route<8>(a, stream) : dispatch_route<32>(a, stream);
}
