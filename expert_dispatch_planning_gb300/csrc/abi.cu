// abi.cu -- host-side pieces of the C ABI shared by every entry point:
// status strings, reading the plan's device status word, launch settings
// (programmatic dependent launch, SM count) and the bounded-wait test hook.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "moe_common.cuh"

namespace {
std::atomic<int> g_skip_tile{-1};
std::atomic<int64_t> g_timeout_ns{1000000000};  // 1 s
}  // namespace

namespace moe_host {

bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("MOE_PDL");
        return v == nullptr || std::strcmp(v, "0") != 0;
    }();
    return on;
}

// SM count of the current device, cached per device (safe for concurrent
// callers); GB300's 152 if the query fails.
int num_sms() {
    constexpr int kFallback = 152;
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices];  // 0: not queried yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kFallback;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached) {
        const int n = cache[dev].load(std::memory_order_relaxed);
        if (n > 0) return n;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kFallback;
    if (cached) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int64_t timeout_ns() { return g_timeout_ns.load(); }
int skip_tile() { return g_skip_tile.load(); }

}  // namespace moe_host

extern "C" MOE_API const char* moe_status_string(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported combination";
        case MOE_ERR_CAPACITY: return "buffer too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case MOE_ERR_DEVICE_INDEX: return "device index out of range";
        case MOE_ERR_WORKSPACE: return "plan workspace not initialised";
        case MOE_ERR_DEVICE_CAPACITY: return "rank row budget exceeded";
        default: return "unknown status";
    }
}

extern "C" MOE_API int moe_get_status(const MoePlanOut* plan, int32_t* device_status, cudaStream_t stream) {
    if (plan == nullptr || plan->status == nullptr || device_status == nullptr) return MOE_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    int32_t host[2] = {0, 0};
    if (cudaMemcpy(host, plan->status, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(plan->status, 0, sizeof(host)) != cudaSuccess) return MOE_ERR_CUDA;
    *device_status = host[0];
    return MOE_OK;
}

extern "C" MOE_API int moe_debug_set_plan_fault(int skip_tile, int64_t timeout_ns) {
    if (skip_tile < -1 || timeout_ns < 0) return MOE_ERR_INVALID_ARG;
    g_skip_tile.store(skip_tile);
    g_timeout_ns.store(timeout_ns > 0 ? timeout_ns : 1000000000);
    return MOE_OK;
}

// Plan reuse (MoonEP MoonEPCommPlan.clone; DeepEP's cached dispatch reuses a
// plan without planning again): a plan is caller-owned and stays valid for
// any number of permute / combine calls; this copies one plan into another
// set of buffers of the same sizes, one asynchronous device copy per array.
extern "C" MOE_API int moe_plan_copy(const MoePlanOut* src, const MoePlanOut* dst, int N, int E, int K, int R,
                                     int alignment, cudaStream_t stream) {
    if (src == nullptr || dst == nullptr || N < 0 || E < 1 || K < 1 || R < 1 || alignment < 1 || E % R != 0)
        return MOE_ERR_INVALID_ARG;
    const int64_t p_cap = moe_plan_capacity_rows(N, E, K, alignment);
    if (p_cap < 0) return MOE_ERR_INVALID_ARG;
    struct Item {
        const void* s;
        void* d;
        size_t bytes;
    } items[] = {
        {src->tokens_per_expert, dst->tokens_per_expert, 4u * E},
        {src->cu_seqlens, dst->cu_seqlens, 4u * (E + 1)},
        {src->zero_fill_ranges, dst->zero_fill_ranges, 8u * E},
        {src->pairs_per_rank, dst->pairs_per_rank, 4u * R},
        {src->tokens_per_rank, dst->tokens_per_rank, 4u * R},
        {src->rank_prefix, dst->rank_prefix, 4u * (R + 1)},
        {src->rank_slot_offsets, dst->rank_slot_offsets, 4u * (R + 1)},
        {src->is_token_in_rank, dst->is_token_in_rank, static_cast<size_t>(N) * R},
        {src->dst, dst->dst, 4u * static_cast<size_t>(N) * K},
        {src->src_of_slot, dst->src_of_slot, 4u * static_cast<size_t>(p_cap)},
        {src->dup_groups, dst->dup_groups, 12u * static_cast<size_t>(N) * (K / 2)},
        {src->dup_loffs, dst->dup_loffs, 4u * static_cast<size_t>(N) * (K - 1)},
        {src->dup_counts, dst->dup_counts, 8u},
        {src->status, dst->status, 16u},
    };
    for (const Item& it : items) {
        if (it.bytes == 0) continue;
        if (it.s == nullptr || it.d == nullptr) return MOE_ERR_INVALID_ARG;
    }
    for (const Item& it : items) {
        if (it.bytes == 0) continue;
        if (cudaMemcpyAsync(it.d, it.s, it.bytes, cudaMemcpyDeviceToDevice, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
