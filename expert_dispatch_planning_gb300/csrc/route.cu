// route.cu -- router top-K kernels for one GPU (sm_103a).
//
// route_topk_kernel: a grid-stride loop over tokens, G lanes per token, the
// next token's logits in flight while route_token (route_core.cuh) picks the
// current token's experts and weights; every shape.
// route_fast_kernel (route_fast.cuh): E = 32 G, sigmoid over groups of 32
// experts or renormalised softmax, selection by approximate keys proved
// exact, the exact router as the per-token fallback; bit-identical output.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "route_fast.cuh"

namespace moe {

template <int G, int V, bool VEC, int KMAX>
__global__ void __launch_bounds__(ROUTE_THREADS) route_topk_kernel(const RouteArgs a) {
    extern __shared__ float s_keys_all[];  // [warps][E], general group-limited path only
    constexpr int TPW = 32 / G;              // tokens per warp
    constexpr int KPL = (KMAX + G - 1) / G;  // winners kept per lane
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane % G;
    const int K = a.K;
    float* s_keys = s_keys_all + warp * a.E;
    pdl_wait();
    pdl_trigger();
    float bias_r[V];  // this lane's experts' bias, the same for every token
    lane_bias<G, V, VEC>(a, sub, bias_r);
    const int64_t step = static_cast<int64_t>(gridDim.x) * (ROUTE_THREADS / 32) * TPW;
    int64_t wtok = (static_cast<int64_t>(blockIdx.x) * (ROUTE_THREADS / 32) + warp) * TPW;
    float nxt[V];
    if (wtok < a.N) load_row<G, V, VEC>(a, wtok + lane / G, sub, nxt);
    for (; wtok < a.N; wtok += step) {
        const int64_t s = wtok + lane / G;
        const bool valid = s < a.N;
        float raw[V];
#pragma unroll
        for (int v = 0; v < V; ++v) raw[v] = nxt[v];
        if (wtok + step < a.N) load_row<G, V, VEC>(a, wtok + step + lane / G, sub, nxt);  // next token in flight

        int my_idx[KPL];
        float num[KPL];
        route_token<G, V, VEC, KMAX>(a, raw, bias_r, valid, lane, sub, s_keys, my_idx, num);

        // ---- store
        if (valid) {
#pragma unroll
            for (int t = 0; t < KPL; ++t) {
                const int k = sub + G * t;
                if (k < K) {
                    a.topk_idx[s * K + k] = my_idx[t];
                    a.topk_w[s * K + k] = num[t];
                }
            }
        }
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

// The selection-by-approximate-keys kernel applies to: E = 32 G for G in
// {4, 8, 16}, K <= 8, and either sigmoid scores with no groups or one group
// per 32 experts and K <= G, or renormalised softmax scores without groups.
// It runs from 16384 tokens on: below that its own gain (about 1 us at 4096
// to 8192 tokens) is smaller than what its longer-lived blocks cost the
// neighbouring plan and row kernels in the route -> plan -> permute ->
// combine chain (2 to 4 us per step measured at those sizes; at 65536 tokens
// it saves 80 us).  MOE_ROUTE_PATH=exact keeps every call on
// route_topk_kernel, MOE_ROUTE_PATH=fast takes the fast kernel at any N.
bool route_fast_shape(const RouteArgs& a) {
    if (a.E % 32 != 0 || a.K > 8) return false;
    const int G = a.E / 32;
    if (G != 4 && G != 8 && G != 16) return false;
    if (a.scoring == MOE_SCORING_SOFTMAX) return a.renormalize && a.n_group == 1;
    if (a.n_group != 1 && a.n_group != G) return false;
    return a.K <= G;
}

constexpr int kRouteFastMinTokens = 16384;

bool route_fast_applies(const RouteArgs& a) {
    const char* env = std::getenv("MOE_ROUTE_PATH");
    if (env != nullptr && std::strcmp(env, "exact") == 0) return false;
    if (!route_fast_shape(a)) return false;
    if (env != nullptr && std::strcmp(env, "fast") == 0) return true;
    return a.N >= kRouteFastMinTokens;
}

template <int G, bool SM>
int launch_route_fast(const RouteArgs& a, cudaStream_t stream) {
    constexpr int tokens_per_block = moe::RF_WARPS * (32 / G);
    const int64_t batches = (static_cast<int64_t>(a.N) + tokens_per_block - 1) / tokens_per_block;
    const size_t smem = sizeof(float) * (32 * G + moe::RF_WARPS * 1024);
    // a wave of resident blocks, the same number of batches for every block
    static std::atomic<int> per_sm_cache{0};  // the same for every GB300; 0: not queried yet
    int per_sm = per_sm_cache.load(std::memory_order_relaxed);
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, moe::route_fast_kernel<G, SM>, moe::RF_THREADS,
                                                          smem) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        per_sm_cache.store(per_sm, std::memory_order_relaxed);
    }
    const int64_t cap = static_cast<int64_t>(moe_host::num_sms()) * per_sm;
    // one wave, or several when a block would get more tokens than its
    // queue for the exact router holds
    int64_t rounds = (batches + cap - 1) / cap;
    rounds = std::min<int64_t>(rounds, moe::RF_DEFER / tokens_per_block);
    const int64_t blocks = (batches + rounds - 1) / rounds;
    // in stream order: started early, its blocks (17 KB of shared memory
    // each) slowed the kernel before it by more than the launch gap it hides
    return moe_host::launch_ordered(moe::route_fast_kernel<G, SM>, dim3(static_cast<unsigned>(blocks)),
                                    dim3(moe::RF_THREADS), smem, stream, a);
}

template <bool SM>
int dispatch_route_fast(const RouteArgs& a, cudaStream_t stream) {
    switch (a.E / 32) {
        case 4: return launch_route_fast<4, SM>(a, stream);
        case 8: return launch_route_fast<8, SM>(a, stream);
        default: return launch_route_fast<16, SM>(a, stream);
    }
}

}  // namespace

extern "C" MOE_API int moe_route_topk(const float* logits, const float* bias, int N, int E, int K,
                                      int scoring, int renormalize, int n_group, int topk_group,
                                      float routed_scaling, int32_t* topk_idx, float* topk_w,
                                      cudaStream_t stream) {
    RouteArgs a;
    const int rc = moe_host::route_args(logits, bias, N, E, K, scoring, renormalize, n_group, topk_group,
                                        routed_scaling, topk_idx, topk_w, &a);
    if (rc != MOE_OK) return rc;
    if (N == 0) return MOE_OK;  // an empty batch: nothing to route, no launch
    if (route_fast_applies(a))
        return a.scoring == MOE_SCORING_SOFTMAX ? dispatch_route_fast<true>(a, stream)
                                                : dispatch_route_fast<false>(a, stream);
    return K <= 8 ? dispatch_route<8>(a, stream) : dispatch_route<32>(a, stream);
}

extern "C" MOE_API int moe_debug_route_sigmoid_error(float* max_abs_err, cudaStream_t stream) {
    if (max_abs_err == nullptr) return MOE_ERR_INVALID_ARG;
    if (cudaMemsetAsync(max_abs_err, 0, sizeof(float), stream) != cudaSuccess) return MOE_ERR_CUDA;
    moe::sigmoid_error_kernel<<<moe_host::num_sms() * 8, 256, 0, stream>>>(reinterpret_cast<uint32_t*>(max_abs_err));
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
