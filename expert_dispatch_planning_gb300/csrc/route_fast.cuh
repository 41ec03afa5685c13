// route_fast.cuh -- the router for E = 32 * G experts (G = 4, 8, 16), sm_103a:
// sigmoid scores over groups of 32 experts (DeepSeek-style group-limited
// routing) and renormalised softmax scores.
//
// The exact router (route_core.cuh) evaluates the fixed-sequence sigmoid for
// every expert and runs K warp-wide arg-max rounds per token; at E = 256 that
// is about 1500 warp instructions per token.  Only the winners' keys decide
// the output, so this kernel selects with cheap approximate keys and proves
// the selection exact afterwards:
//
//   1. G lanes per token, lane `sub` owns the 32 contiguous experts of group
//      `sub`.  Approximate key a = rcp.approx(1 + ex2.approx(-x log2 e)) + b,
//      within RF_DELTA_SIGMA of the fixed sigmoid (re-measured over every
//      fp32 input by moe_debug_route_sigmoid_error) plus one key rounding of
//      the exact key.  The expert's lane-local index is packed into the 5
//      low bits of a, so that packed keys are distinct within a lane; a
//      7-deep min/max network keeps the lane's seven largest (its first
//      level propagates NaN, which marks a NaN logit).
//   2. Group score = sum of the lane's two largest packed keys; the
//      topk_group best groups (rank by shuffles within the token) are kept.
//   3. K + 1 rounds of arg-max over the kept lanes' list heads (max by xor
//      shuffles, ties to the lowest lane); the K-th and (K+1)-th maxima and
//      the groups on both sides of the topk_group boundary must be separated
//      by more than twice the packed keys' error bound.  Then no exact key
//      can reorder across either boundary, and the exact top-K set and the
//      exact kept groups are the approximate ones.
//   4. Winners whose consecutive round maxima are separated by the same
//      margin are already in exact order; otherwise (sigmoid) their exact
//      keys (the exact router's fixed sigmoid) sort them, descending, ties
//      to the lower index.  The weights are computed in sorted position with
//      the exact router's arithmetic and summation order, so the output is
//      bit-identical to it.
//   5. A token that fails a check (a margin, a lane that ran out of its
//      seven candidates, a NaN logit; with softmax scores any non-finite
//      one) is routed by a whole warp with the exact router's route_token;
//      so is every token when a bias is not finite or exceeds 2^20 in
//      magnitude.  Such tokens are queued in shared memory and routed at the
//      end of the block, their logits read again from global memory, so
//      that no warp holds its batch loop on a slow token.  The margins scale
//      with the largest |bias| (the keys' ulp).  An infinite logit needs no
//      exception with sigmoid scores: its approximate key is within the
//      bound like any other (the sweep covers every non-NaN input).
//   Softmax: the key is the logit, so a packed key is within 2^-18 of it
//   (relative); the margins are relative too, and out-of-order winners (a
//   near-tie inside the top K) go to the exact router.  With 4 lanes per
//   token a lane holds winners 2*sub and 2*sub + 1, which keeps the
//   normaliser's summation tree that of the exact router.
//
// Logits are staged per warp in shared memory with 16-byte cp.async copies
// (one 4 KB batch per warp; eight blocks per SM hide the load); each lane
// reads its 128-byte group in a rotated chunk order so that the eight lanes
// of a token hit eight different bank quads.
#pragma once

#include "route_core.cuh"

namespace moe {

// ---------------------------------------------------------------- approximate sigmoid
// Hardware approximations, used only to choose candidates.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sigmoid_approx(float x) {
    return rcp_approx(__fadd_rn(1.0f, ex2_approx(__fmul_rn(x, -0x1.715476p+0f))));
}

// |sigmoid_approx(x) - sigmoid_f32(x)| <= RF_DELTA_SIGMA for every fp32 x
// (about twice the largest difference over all 2^32 inputs; the GPU tests
// re-run that sweep against half of this constant).
constexpr float RF_DELTA_SIGMA = 0x1p-20f;

// Separation demanded at the two boundaries, for keys of magnitude <= M
// (M bounds |sigmoid| + max|bias| with room for the approximation).  With
// u = the fp32 ulp at M: a packed key is within eps = DELTA_SIGMA + u (the
// two key sums' roundings, half an ulp each) + 31 u (the replaced low bits)
// of the exact key; a group sum of two packed keys is within 2 eps + 2 u
// (both sums' roundings at 2M) of the exact group score.  The checks demand
// twice these, times 17/16 for the subtraction that tests them.
struct FastMargins {
    float k, g;
};
__device__ __forceinline__ FastMargins fast_margins(float bmax) {
    const float M = __fadd_ru(__fadd_ru(1.0f, bmax), 0x1p-19f);
    const float u = __uint_as_float(((__float_as_uint(M) >> 23) - 23u) << 23);  // M >= 1: 2^(exp(M) - 23)
    const float eps = __fadd_ru(RF_DELTA_SIGMA, __fmul_ru(32.0f, u));
    FastMargins m;
    m.k = __fmul_ru(2.125f, eps);
    m.g = __fmul_ru(2.125f, __fadd_ru(__fmul_ru(2.0f, eps), __fmul_ru(2.0f, u)));
    return m;
}
constexpr int RF_D = 7;        // candidates kept per lane
constexpr int RF_DEFER = 512;  // tokens a block may hand to the exact router: every token
                               // of the block (the launch keeps blocks within this)
constexpr int RF_THREADS = 128;
constexpr int RF_WARPS = RF_THREADS / 32;

// max that returns NaN when either input is NaN (fmaxf drops a NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Separation check of two packed keys hi >= lo.  Sigmoid keys: more than
// the absolute margin m.  Softmax keys (the logits themselves, approximate
// only in the 5 replaced low bits, i.e. within 2^-18 relative): more than
// 2^-16 (|hi| + |lo|) plus room for subnormals.
template <bool SM>
__device__ __forceinline__ bool separated(float hi, float lo, float m) {
    if constexpr (SM) {
        return __fsub_rn(hi, lo) > __fmaf_rn(0x1p-16f, __fadd_rn(fabsf(hi), fabsf(lo)), 0x1p-120f);
    } else {
        return __fsub_rn(hi, lo) > m;
    }
}

// One token of the current batch: the segment of G lanes starting at
// lane t*G.  SM: softmax scores (key = logit, no groups, renormalised
// weights); else sigmoid + bias with optional groups of 32.  Lane `sub`
// holds winners k = KPL*sub + j, j < KPL (KPL = 2 when K > G).  Returns
// true when the token needs the exact router.
template <int G, bool SM>
__device__ __forceinline__ bool route_fast_token(const RouteArgs& a, const float* row, const float* s_bias,
                                                 bool fast_ok, FastMargins mg, int sub, int64_t s, bool valid) {
    constexpr unsigned SEGMASK = G == 32 ? 0xffffffffu : ((1u << G) - 1u);
    constexpr int KPL = (SM && G < 8) ? 2 : 1;  // winners per lane (K <= 8; sigmoid: K <= G)
    const int lane = threadIdx.x & 31;
    const int segbase = lane & ~(G - 1);
    const int K = a.K;
    const bool has_bias = a.bias != nullptr;

    // ---- 1. packed approximate keys, the lane's RF_D largest
    float L[RF_D];
#pragma unroll
    for (int d = 0; d < RF_D; ++d) L[d] = -INFINITY;
    float nan_chk = 0.0f;  // softmax: stays 0 unless a logit is NaN or infinite
    const float* grp = row + 32 * sub;
    const float* gb = s_bias + 32 * sub;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = (i + sub) & 7;  // rotated 16-byte chunk: no bank conflicts
        const float4 q = *reinterpret_cast<const float4*>(grp + 4 * c);
        const float xs[4] = {q.x, q.y, q.z, q.w};
        float bs[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (!SM) {
            const float4 bq = *reinterpret_cast<const float4*>(gb + 4 * c);
            bs[0] = bq.x;
            bs[1] = bq.y;
            bs[2] = bq.z;
            bs[3] = bq.w;
        }
        const uint32_t jbase = 31u - 4u * static_cast<uint32_t>(c);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            // sigmoid: a NaN logit gives a NaN key (an infinite one a key
            // within the bound); softmax keys are the logits, checked finite
            if constexpr (SM) nan_chk = __fmaf_rn(xs[u], 0.0f, nan_chk);
            const float ak = SM ? xs[u] : __fadd_rn(sigmoid_approx(xs[u]), bs[u]);
            const float v = __uint_as_float((__float_as_uint(ak) & ~31u) | (jbase - static_cast<uint32_t>(u)));
            // insertion into the sorted list: the new d-th largest is
            // max(L[d], min(L[d-1], v)); a NaN stays in L[0] from then on
            float n[RF_D];
            n[0] = max_nan(L[0], v);
#pragma unroll
            for (int d = 1; d < RF_D; ++d) n[d] = fmaxf(L[d], fminf(L[d - 1], v));
#pragma unroll
            for (int d = 0; d < RF_D; ++d) L[d] = n[d];
        }
    }

    // ---- 2. group selection (sigmoid)
    bool kept = true;
    bool fail = !fast_ok || L[0] != L[0] || nan_chk != 0.0f;
    if (!SM && a.n_group > 1 && a.topk_group < G) {
        const float S = __fadd_rn(L[0], L[1]);
        int rank = 0;
#pragma unroll
        for (int d = 1; d < G; ++d) {
            const int o = (sub + d) & (G - 1);
            const float So = __shfl_sync(FULL_MASK, S, o, G);
            rank += (So > S || (So == S && o < sub)) ? 1 : 0;
        }
        kept = rank < a.topk_group;
        float kmin = kept ? S : INFINITY;
        float nmax = kept ? -INFINITY : S;
#pragma unroll
        for (int off = 1; off < G; off <<= 1) {
            kmin = fminf(kmin, __shfl_xor_sync(FULL_MASK, kmin, off, G));
            nmax = fmaxf(nmax, __shfl_xor_sync(FULL_MASK, nmax, off, G));
        }
        if (!(__fsub_rn(kmin, nmax) > mg.g)) fail = true;
    }

    // ---- 3. K + 1 rounds of arg-max over the kept lanes' heads
    int my_e[KPL];         // winners k = KPL * sub + j
#pragma unroll
    for (int j = 0; j < KPL; ++j) my_e[j] = 0;
    float mK = 0.f, mK1 = 0.f, mprev = 0.f;
    bool ordered = true;   // consecutive winners separated by the margin
    int popped = 0;
    bool exhausted = false;
    if (!kept) {
#pragma unroll
        for (int d = 0; d < RF_D; ++d) L[d] = -INFINITY;
    }
#pragma unroll
    for (int r = 0; r <= 8; ++r) {
        if (r > K) break;
        float mx = L[0];
#pragma unroll
        for (int off = 1; off < G; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, off, G));
        const uint32_t eq = (__ballot_sync(FULL_MASK, L[0] == mx) >> segbase) & SEGMASK;
        const int w = __ffs(eq) - 1;  // lowest lane holding the maximum
        if (r == K - 1) mK = mx;
        if (r == K) mK1 = mx;
        if (r > 0 && r < K && !separated<SM>(mprev, mx, mg.k)) ordered = false;
        mprev = mx;
        if (r < K) {
            if (sub == r / KPL) my_e[r % KPL] = 32 * w + 31 - static_cast<int>(__float_as_uint(mx) & 31u);
            if (sub == w) {
#pragma unroll
                for (int d = 0; d < RF_D - 1; ++d) L[d] = L[d + 1];
                L[RF_D - 1] = -INFINITY;
                ++popped;
                if (popped == RF_D) exhausted = true;  // its next key is unknown
            }
        }
    }
    if (exhausted) fail = true;
    if (!separated<SM>(mK, mK1, mg.k)) fail = true;
    if (SM && !ordered) fail = true;  // softmax: out-of-order winners go to the exact router
    fail = ((__ballot_sync(FULL_MASK, fail) >> segbase) & SEGMASK) != 0u;

    // ---- 4. the winners in exact order.  Consecutive round maxima more
    // than the margin apart are in exact-key order already; otherwise
    // (sigmoid) the winners' exact keys sort them (descending, ties to the
    // lower index) -- for the whole warp when any token needs it.
    int ek[KPL];
    float xk[KPL];
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
        const bool win = KPL * sub + j < K;
        ek[j] = win ? (my_e[j] & (32 * G - 1)) : 0x7fffffff;  // always in range
        xk[j] = win ? row[ek[j] & (32 * G - 1)] : 0.f;
    }
    if constexpr (!SM) {
        const int e = ek[0];
        const float x = xk[0];
        const bool need_sort = ((__ballot_sync(FULL_MASK, !ordered) >> segbase) & SEGMASK) != 0u;
        if (__any_sync(FULL_MASK, need_sort)) {
            uint32_t okey = 0u;
            if (sub < K) {
                const float sg = sigmoid_f32(x);
                okey = order_key(has_bias ? __fadd_rn(sg, s_bias[e]) : sg);
            }
            int rank = 0;
#pragma unroll
            for (int d = 1; d < G; ++d) {
                const int o = (sub + d) & (G - 1);
                const uint32_t ko = __shfl_sync(FULL_MASK, okey, o, G);
                const int eo = __shfl_sync(FULL_MASK, e, o, G);
                rank += (ko > okey || (ko == okey && eo < e)) ? 1 : 0;
            }
            int src = 0;  // the lane whose winner sorts to position `sub`
#pragma unroll
            for (int d = 0; d < G; ++d) {
                const int rd = __shfl_sync(FULL_MASK, rank, d, G);
                if (rd == sub) src = d;
            }
            const float xs = __shfl_sync(FULL_MASK, x, src, G);
            const int es = __shfl_sync(FULL_MASK, e, src, G);
            if (need_sort) {
                xk[0] = xs;
                ek[0] = es;
            }
        }
    }

    // ---- 5. weights with the exact router's arithmetic; with the winners
    // of lane sub at k = KPL*sub + j, the within-lane sums and the xor
    // butterfly add in the exact router's tree order
    float num[KPL], shi = 0.f, slo = 0.f;
    bool tiny_tok = false;
    if constexpr (SM) {
        const float top = __shfl_sync(FULL_MASK, xk[0], 0, G);  // the row maximum
#pragma unroll
        for (int j = 0; j < KPL; ++j) {
            num[j] = 0.f;
            if (KPL * sub + j < K) {
                num[j] = exp_diff(xk[j], top);
                ff_add(shi, slo, num[j], 0.f);
            }
        }
    } else {
        num[0] = 0.f;
        if (sub < K) {
            num[0] = sigmoid_weight(xk[0]);
            if (a.renormalize && num[0] >= 0x1p-100f) ff_add(shi, slo, num[0], 0.f);
        }
        tiny_tok = ((__ballot_sync(FULL_MASK, sub < K && num[0] < 0x1p-100f) >> segbase) & SEGMASK) != 0u;
        if (__any_sync(FULL_MASK, tiny_tok)) {
            double sd = 0.0;
            if (sub < K) {
                const double ex = exp(-fabs(static_cast<double>(xk[0])));
                sd = xk[0] >= 0.f ? 1.0 / (1.0 + ex) : ex / (1.0 + ex);
            }
            double den = sd;
#pragma unroll
            for (int off = 1; off < G; off <<= 1) den += __shfl_xor_sync(FULL_MASK, den, off, G);
            const double scale = a.renormalize ? static_cast<double>(a.scaling) / den : a.scaling;
            if (tiny_tok) num[0] = static_cast<float>(sd * scale);
        }
    }
    // (every lane takes part in the shuffles; tokens on the fp64 path keep
    // the value above)
#pragma unroll
    for (int off = 1; off < G; off <<= 1) {
        const float oh = __shfl_xor_sync(FULL_MASK, shi, off, G);
        const float ol = __shfl_xor_sync(FULL_MASK, slo, off, G);
        ff_add(shi, slo, oh, ol);
    }
    if (!tiny_tok) {
        if (SM || a.renormalize) {
            const float q = __fdiv_rn(a.scaling, shi);
            const float qc = __fmaf_rn(-q, __fdiv_rn(slo, shi), q);
#pragma unroll
            for (int j = 0; j < KPL; ++j) num[j] = __fmul_rn(num[j], qc);
        } else {
            num[0] = __fmul_rn(num[0], a.scaling);
        }
    }
    if (valid && !fail) {
#pragma unroll
        for (int j = 0; j < KPL; ++j) {
            const int k = KPL * sub + j;
            if (k < K) {
                a.topk_idx[s * K + k] = ek[j];
                a.topk_w[s * K + k] = num[j];
            }
        }
    }
    return fail;
}

// G lanes per token (E = 32 G), 32 / G tokens per warp per batch; SM:
// softmax scores.
template <int G, bool SM>
__global__ void __launch_bounds__(RF_THREADS, 8) route_fast_kernel(const RouteArgs a) {
    extern __shared__ __align__(16) float s_mem[];  // bias [E], then [warps][1024] logits
    constexpr int TPW = 32 / G;
    constexpr int E = 32 * G;
    constexpr int V = E / 32;  // values per lane in the exact router's layout
    constexpr int STAGE = TPW * E;  // floats per batch (always 1024)
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane & (G - 1);
    const int t = lane / G;
    const int K = a.K;
    float* s_bias = s_mem;
    float* stage = s_mem + E + warp * STAGE;

    const int64_t step = static_cast<int64_t>(gridDim.x) * RF_WARPS * TPW;
    int64_t tok0 = (static_cast<int64_t>(blockIdx.x) * RF_WARPS + warp) * TPW;
    auto issue = [&](int64_t first) {
        const int64_t n = min(static_cast<int64_t>(TPW), static_cast<int64_t>(a.N) - first);
        const float* srcp = a.logits + first * E;
        const int chunks = static_cast<int>(n) * (E / 4);
        for (int c = lane; c < chunks; c += 32) cp_async_16(stage + 4 * c, srcp + 4 * c);
        cp_async_commit();
    };
    pdl_wait();
    pdl_trigger();
    if (tok0 < a.N) issue(tok0);  // in flight while the bias is read

    // the bias in shared memory (zero without one) and the largest |bias|
    float bmax = 0.0f;
    bool finite = true;
    for (int e = threadIdx.x; e < E; e += RF_THREADS) {
        const float b = a.bias != nullptr ? __ldg(a.bias + e) : 0.0f;
        s_bias[e] = b;
        if (!(fabsf(b) <= 0x1p20f)) finite = false;
        bmax = fmaxf(bmax, fabsf(b));
    }
    const bool fast_ok = __syncthreads_and(finite) != 0;
    __shared__ float s_bmax[RF_WARPS];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(FULL_MASK, bmax, off));
    if (lane == 0) s_bmax[warp] = bmax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < RF_WARPS; ++w) bmax = fmaxf(bmax, s_bmax[w]);
    const FastMargins mg = fast_margins(fast_ok ? bmax : 0.0f);

    // tokens that failed a check, routed exactly after the batch loop (the
    // launch gives a block at most RF_DEFER tokens, so the queue never fills)
    __shared__ int32_t s_defer[RF_DEFER];
    __shared__ int s_ndefer;
    if (threadIdx.x == 0) s_ndefer = 0;
    __syncthreads();

    for (; tok0 < a.N; tok0 += step) {
        float* cur = stage;
        cp_async_wait_0();
        __syncwarp();
        const int64_t s = tok0 + t;
        const bool valid = s < a.N;
        const float* row = cur + t * E;  // rows past N hold stale data; nothing is stored for them
        const bool fail = route_fast_token<G, SM>(a, row, s_bias, fast_ok, mg, sub, s, valid);

        // tokens that failed a check: queued for the end of the block (N < 2^31)
        const bool queue = fail && valid;
        const uint32_t qmask = __ballot_sync(FULL_MASK, queue && sub == 0);
        if (qmask != 0u) {
            int base = 0;
            if (lane == 0) base = atomicAdd(&s_ndefer, __popc(qmask));
            base = __shfl_sync(FULL_MASK, base, 0);
            const int slot = base + __popc(qmask & ((1u << lane) - 1u));
            if (queue && sub == 0 && slot < RF_DEFER) s_defer[slot] = static_cast<int32_t>(s);
        }
        __syncwarp();  // every lane is done with the stage before it is refilled
        if (tok0 + step < a.N) issue(tok0 + step);
    }

    // the queued tokens, a warp each, by the exact router; their logits
    // read again from global memory
    __syncthreads();
    const int nq = min(s_ndefer, RF_DEFER);
    for (int i = warp; i < nq; i += RF_WARPS) {
        const int64_t st = s_defer[i];
        const float* lrow = a.logits + st * E;
        float raw[V], bias32[V];
#pragma unroll
        for (int j = 0; j < V / 4; ++j) {
            const float4 q = *reinterpret_cast<const float4*>(lrow + 4 * (lane + 32 * j));
            raw[4 * j + 0] = q.x;
            raw[4 * j + 1] = q.y;
            raw[4 * j + 2] = q.z;
            raw[4 * j + 3] = q.w;
        }
        lane_bias<32, V, true>(a, lane, bias32);
        int my_idx[1];
        float num[1];
        route_token<32, V, true, 8>(a, raw, bias32, true, lane, lane, nullptr, my_idx, num);
        if (lane < K) {
            a.topk_idx[st * K + lane] = my_idx[0];
            a.topk_w[st * K + lane] = num[0];
        }
    }
}

// Every fp32 bit pattern x (NaN skipped): max |sigmoid_approx(x) -
// sigmoid_f32(x)| into *max_err (as float bits; zero it first).
__global__ void sigmoid_error_kernel(uint32_t* max_err) {
    uint32_t worst = 0u;
    const uint64_t n = uint64_t(1) << 32;
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const float x = __uint_as_float(static_cast<uint32_t>(i));
        if (x != x) continue;
        const float d = fabsf(__fsub_rn(sigmoid_approx(x), sigmoid_f32(x)));
        worst = max(worst, __float_as_uint(d));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) worst = max(worst, __shfl_xor_sync(FULL_MASK, worst, off));
    if ((threadIdx.x & 31) == 0) atomicMax(max_err, worst);
}

}  // namespace moe
