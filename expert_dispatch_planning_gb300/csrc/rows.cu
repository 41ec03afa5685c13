// rows.cu -- bandwidth-bound row movement for one GPU (sm_103a).
//
// moe_permute: every pair's token row goes to its slot of the
// expert-contiguous buffer (DeepEP csrc/kernels/intranode.cu, dispatch: a
// warp copies each token's hidden row with 16-byte vectors), and the padding
// rows named by the plan's zero-fill ranges (MoonEP moonep/planning.py) are
// written as zeros.  Each x row is read from HBM once and fanned out K times
// by the bulk-copy engine: one cp.async.bulk global->shared load per group of
// tokens (completion on an mbarrier, together with the 4-byte cp.async loads
// of the group's dst entries), then one cp.async.bulk shared->global store
// per pair.  A single-warp CTA keeps a ring of stages in flight; many small
// CTAs share an SM.
//
// moe_combine: out[s] = bf16(sum_k w[s,k] * y[slot(s,k)]) accumulated in
// fp32, one fused multiply-add per pair in k order, rounded to nearest even
// (DeepEP combine: fp32 accumulation of the gathered rows, cast back to the
// dtype; here weighted).  A warp per token, each lane owning 16-byte chunks,
// all K row loads of a chunk issued before the arithmetic.
#include <cuda_bf16.h>

#include "moe_common.cuh"

namespace moe {

// ---------------------------------------------------------------- permute
struct PermuteArgs {
    const uint16_t* x;
    uint16_t* out;
    const int32_t* dst;
    const int32_t* zfr;
    int32_t* status;
    int N, H, K, E, alignment;
    int64_t p_cap;
    int G;        // tokens per stage
    int stages;   // ring depth
    int64_t n_groups;
    uint32_t stage_bytes;  // G * row bytes rounded up to 128
    uint32_t slots_bytes;  // stages * G * K * 4 rounded up to 128
    int64_t timeout_ns;
    int early_x;  // load the first stages' x rows before waiting on the predecessor kernel
};

__global__ void __launch_bounds__(32) permute_kernel(const PermuteArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);                  // [stages]
    int32_t* slots = reinterpret_cast<int32_t*>(smem + 128);             // [stages][G*K]
    uint8_t* rows = smem + 128 + a.slots_bytes;                          // [stages][stage_bytes]

    const int lane = threadIdx.x;
    const int K = a.K, G = a.G;
    const uint32_t row_bytes = static_cast<uint32_t>(a.H) * 2u;
    const int64_t H = a.H;
    if (lane == 0) {
        for (int st = 0; st < a.stages; ++st) mbar_init(&bar[st], 33);
        fence_mbar_init();
    }
    __syncwarp();

    const int64_t g_begin = blockIdx.x * a.n_groups / gridDim.x;
    const int64_t g_end = (blockIdx.x + 1) * a.n_groups / gridDim.x;
    const int64_t n_mine = g_end - g_begin;

    // A stage completes when its x rows (one bulk load, lane 0's arrive with
    // the byte count) and its dst entries (4-byte cp.async loads, one
    // no-increment arrive per lane) have landed: 33 arrivals.
    auto issue_x = [&](int64_t i) {  // x rows of group g_begin + i into stage i % stages
        if (lane == 0) {
            const int st = static_cast<int>(i % a.stages);
            const int64_t tok0 = (g_begin + i) * G;
            const int ntok = static_cast<int>(min(static_cast<int64_t>(G), static_cast<int64_t>(a.N) - tok0));
            const uint32_t bytes = static_cast<uint32_t>(ntok) * row_bytes;
            mbar_arrive_expect_tx(&bar[st], bytes);
            bulk_g2s(rows + static_cast<size_t>(st) * a.stage_bytes, a.x + tok0 * H, bytes, &bar[st]);
        }
    };
    auto issue_dst = [&](int64_t i) {  // the group's dst entries
        const int st = static_cast<int>(i % a.stages);
        const int64_t tok0 = (g_begin + i) * G;
        const int ntok = static_cast<int>(min(static_cast<int64_t>(G), static_cast<int64_t>(a.N) - tok0));
        const int npairs = ntok * K;
        int32_t* sl = slots + st * G * K;
        for (int p = lane; p < npairs; p += 32) cp_async_4(sl + p, a.dst + tok0 * K + p);
        cp_async_mbar_arrive_noinc(&bar[st]);
    };
    auto issue = [&](int64_t i) {
        issue_dst(i);
        issue_x(i);
    };

    // x does not depend on the plan: with early_x the first stages' rows
    // are requested while the previous kernel (normally the plan) still runs
    int64_t issued = 0;
    if (a.early_x)
        for (; issued < a.stages && issued < n_mine; ++issued) issue_x(issued);

    pdl_wait();
    if (ld_volatile_s32(a.status) != 0) {  // no valid plan to move rows by
        // complete the prefetched stages and let their rows land before the
        // CTA releases its shared memory
        for (int64_t j = 0; j < issued; ++j) cp_async_mbar_arrive_noinc(&bar[j]);
        for (int64_t j = 0; j < issued; ++j) mbar_wait_bounded(&bar[j], 0u, static_cast<uint64_t>(a.timeout_ns));
        return;
    }
    for (int64_t j = 0; j < issued; ++j) issue_dst(j);
    for (; issued < a.stages && issued < n_mine; ++issued) issue(issued);

    bool failed = false;
    int64_t i = 0;
    for (; i < n_mine; ++i) {
        const int st = static_cast<int>(i % a.stages);
        const uint32_t parity = static_cast<uint32_t>((i / a.stages) & 1);
        if (!mbar_wait_bounded(&bar[st], parity, static_cast<uint64_t>(a.timeout_ns))) {
            if (lane == 0) record_error(a.status, MOE_ERR_DEVICE_TIMEOUT, blockIdx.x);
            failed = true;
            break;
        }
        const int64_t tok0 = (g_begin + i) * G;
        const int ntok = static_cast<int>(min(static_cast<int64_t>(G), static_cast<int64_t>(a.N) - tok0));
        const int npairs = ntok * K;
        const int32_t* sl = slots + st * G * K;
        const uint8_t* stage = rows + static_cast<size_t>(st) * a.stage_bytes;
        for (int p = lane; p < npairs; p += 32) {
            const int32_t raw = raw_slot(sl[p]);
            if (raw < 0 || static_cast<int64_t>(raw) >= a.p_cap) {
                record_error(a.status, MOE_ERR_DEVICE_INDEX, raw);
                continue;
            }
            bulk_s2g(a.out + static_cast<int64_t>(raw) * H, stage + static_cast<size_t>(p / K) * row_bytes,
                     row_bytes);
        }
        bulk_commit();
        if (i >= 1) {
            bulk_wait_read<1>();  // stores of group i-1 have left its stage
            __syncwarp();
            if (issued < n_mine) {
                issue(issued);
                ++issued;
            }
        }
    }
    // The next kernel (normally the combine, whose CTAs fill whole SMs) is
    // let in only once this CTA's rows are on their way: dependents resident
    // early slowed the last CTAs' stages (measured: up to 8% of a large step).
    pdl_trigger();
    bulk_wait_read<0>();
    __syncwarp();
    if (failed) {
        // let every load still in flight land before the CTA releases its smem
        for (int64_t j = i + 1; j < issued; ++j) {
            const int st = static_cast<int>(j % a.stages);
            mbar_wait_bounded(&bar[st], static_cast<uint32_t>((j / a.stages) & 1),
                              static_cast<uint64_t>(a.timeout_ns));
        }
        return;
    }

    // ---- padding rows: bulk stores from one zeroed stage
    if (a.alignment > 1) {
        uint4* z = reinterpret_cast<uint4*>(rows);
        for (uint32_t b = lane; b < row_bytes / 16; b += 32) z[b] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncwarp();
        const int per = a.alignment - 1;
        const int64_t virt = static_cast<int64_t>(a.E) * per;
        for (int64_t v = static_cast<int64_t>(blockIdx.x) * 32 + lane; v < virt;
             v += static_cast<int64_t>(gridDim.x) * 32) {
            const int e = static_cast<int>(v / per);
            const int j = static_cast<int>(v - static_cast<int64_t>(e) * per);
            const int32_t cnt = __ldg(a.zfr + 2 * e + 1);
            if (j >= cnt) continue;
            const int64_t row = static_cast<int64_t>(__ldg(a.zfr + 2 * e)) + j;
            if (row < 0 || row >= a.p_cap) {
                record_error(a.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(row));
                continue;
            }
            bulk_s2g(a.out + row * H, rows, row_bytes);
        }
        bulk_commit();
        bulk_wait_read<0>();
    }
}

// ---------------------------------------------------------------- combine
struct CombineArgs {
    const uint16_t* y;
    const float* w;
    const int32_t* dst;
    uint16_t* out;
    int32_t* status;
    int N, K, H;
    int64_t p_cap;
};

constexpr int COMBINE_THREADS = 256;

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void fma_row(float (&acc)[8], float w, const uint4& v) {
    acc[0] = __fmaf_rn(w, bf_lo(v.x), acc[0]);
    acc[1] = __fmaf_rn(w, bf_hi(v.x), acc[1]);
    acc[2] = __fmaf_rn(w, bf_lo(v.y), acc[2]);
    acc[3] = __fmaf_rn(w, bf_hi(v.y), acc[3]);
    acc[4] = __fmaf_rn(w, bf_lo(v.z), acc[4]);
    acc[5] = __fmaf_rn(w, bf_hi(v.z), acc[5]);
    acc[6] = __fmaf_rn(w, bf_lo(v.w), acc[6]);
    acc[7] = __fmaf_rn(w, bf_hi(v.w), acc[7]);
}

__device__ __forceinline__ uint4 pack_row(const float (&acc)[8]) {
    return make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                      pack_bf16x2(acc[6], acc[7]));
}

// KT > 0: K fixed at compile time, U chunks per lane per step with all
// U*KT loads in flight.  KT == 0: any K <= 32, one row at a time.
template <int KT, int U>
__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const CombineArgs a) {
    pdl_wait();
    pdl_trigger();
    if (ld_volatile_s32(a.status) != 0) return;

    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * COMBINE_THREADS + threadIdx.x) >> 5;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (COMBINE_THREADS / 32);
    const int K = KT > 0 ? KT : a.K;
    const int nvec = a.H / 8;
    const int64_t H = a.H;

    for (int64_t s = warp_id; s < a.N; s += warps) {
        int32_t my_raw = 0;
        float my_w = 0.f;
        bool bad = false;
        if (lane < K) {
            my_raw = raw_slot(__ldg(a.dst + s * K + lane));
            my_w = __ldg(a.w + s * K + lane);
            if (my_raw < 0 || static_cast<int64_t>(my_raw) >= a.p_cap) bad = true;
        }
        if (__any_sync(FULL_MASK, bad)) {
            if (bad) record_error(a.status, MOE_ERR_DEVICE_INDEX, my_raw);
            continue;
        }
        uint4* out_row = reinterpret_cast<uint4*>(a.out + s * H);
        if constexpr (KT > 0) {
            const uint4* rows[KT];
            float wk[KT];
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                rows[k] = reinterpret_cast<const uint4*>(a.y + static_cast<int64_t>(__shfl_sync(FULL_MASK, my_raw, k)) * H);
                wk[k] = __shfl_sync(FULL_MASK, my_w, k);
            }
            for (int c0 = lane; c0 < nvec; c0 += 32 * U) {
                uint4 v[U][KT];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + 32 * u;
#pragma unroll
                    for (int k = 0; k < KT; ++k)
                        if (c < nvec) v[u][k] = ld_stream_v4(rows[k] + c);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + 32 * u;
                    if (c >= nvec) continue;
                    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < KT; ++k) fma_row(acc, wk[k], v[u][k]);
                    st_v4(out_row + c, pack_row(acc));
                }
            }
        } else {
            // shuffles stay in converged code: the chunk loop runs the same
            // trip count on every lane and predicates the memory accesses
            for (int c0 = 0; c0 < nvec; c0 += 32) {
                const int c = c0 + lane;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int k = 0; k < K; ++k) {
                    const int32_t raw = __shfl_sync(FULL_MASK, my_raw, k);
                    const float wv = __shfl_sync(FULL_MASK, my_w, k);
                    if (c < nvec) {
                        const uint4 v =
                            ld_stream_v4(reinterpret_cast<const uint4*>(a.y + static_cast<int64_t>(raw) * H) + c);
                        fma_row(acc, wv, v);
                    }
                }
                if (c < nvec) st_v4(out_row + c, pack_row(acc));
            }
        }
    }
}

}  // namespace moe

// ---------------------------------------------------------------- host
namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return v ? std::atoi(v) : dflt;
}

constexpr size_t kSmemPerSm = 227 * 1024;

}  // namespace

extern "C" MOE_API int moe_permute(const uint16_t* x, int N, int H, int K, int E, int alignment,
                                   const MoePlanOut* plan, uint16_t* permuted, int flags, cudaStream_t stream) {
    // N = 0 (an empty batch): no rows to move and, with every expert empty,
    // no padding rows to zero; nothing is written, so x, dst and permuted
    // (E * (alignment - 1) rows, none when alignment is 1) may be null
    if (plan == nullptr || plan->zero_fill_ranges == nullptr || plan->status == nullptr ||
        (N > 0 && (x == nullptr || permuted == nullptr || plan->dst == nullptr)))
        return MOE_ERR_INVALID_ARG;
    if ((flags & ~MOE_PERMUTE_EARLY_X) != 0) return MOE_ERR_INVALID_ARG;
    if (N < 0 || K < 1 || K > 32 || E < 1 || E > 1024 || K > E || alignment < 1 || H < 8 || H % 8 != 0)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(permuted, 16) || !aligned(plan->dst, 4)) return MOE_ERR_INVALID_ARG;
    const int64_t p_cap = moe_plan_capacity_rows(N, E, K, alignment);
    if (p_cap < 0 || p_cap >= (int64_t(1) << 31) - 1) return MOE_ERR_INVALID_ARG;
    const int64_t row_bytes = static_cast<int64_t>(H) * 2;
    if (row_bytes > 96 * 1024) return MOE_ERR_UNSUPPORTED;
    if (N == 0) return MOE_OK;

    moe::PermuteArgs a;
    a.x = x;
    a.out = permuted;
    a.dst = plan->dst;
    a.zfr = plan->zero_fill_ranges;
    a.status = plan->status;
    a.N = N;
    a.H = H;
    a.K = K;
    a.E = E;
    a.alignment = alignment;
    a.p_cap = p_cap;
    // Stages of ~32 KB and a grid of 48 CTAs per SM, each CTA's ring no
    // deeper than the groups it gets: where a CTA gets one or two groups
    // several CTAs are resident per SM, each an independent stream, and the
    // block scheduler balances them to the end; where CTAs get many groups
    // one deep ring per SM keeps the bytes in flight.  Chosen on GB300 by
    // whole-step time (route, plan, permute, combine) over 16-64 KB stages
    // and 6-64 CTAs per SM: 1-9% faster steps than 6 CTAs per SM on the four
    // larger workloads.
    const int64_t target = env_int("MOE_PERMUTE_STAGE_BYTES", 32768);
    int64_t G = target / row_bytes;
    if (G < 1) G = 1;
    if (G > 64) G = 64;
    // small batches: at least two groups per SM so every SM moves rows
    const int64_t spread = (static_cast<int64_t>(N) + 2 * moe_host::num_sms() - 1) / (2 * moe_host::num_sms());
    if (G > spread) G = spread < 1 ? 1 : spread;
    if (G > N) G = N;
    a.G = static_cast<int>(G);
    a.stage_bytes = static_cast<uint32_t>((G * row_bytes + 127) / 128 * 128);
    int stages = env_int("MOE_PERMUTE_STAGES", 16);
    if (stages < 2) stages = 2;
    if (stages > 16) stages = 16;  // 16 mbarriers fit the 128-byte header
    auto slots_for = [&](int st) {
        return static_cast<uint32_t>((static_cast<int64_t>(st) * G * K * 4 + 127) / 128 * 128);
    };
    while (stages > 2 && 128 + slots_for(stages) + static_cast<size_t>(stages) * a.stage_bytes > kSmemPerSm) --stages;
    a.stages = stages;
    a.slots_bytes = slots_for(stages);
    a.n_groups = (N + G - 1) / G;
    a.timeout_ns = moe_host::timeout_ns();
    a.early_x = (flags & MOE_PERMUTE_EARLY_X) != 0 ? 1 : 0;
    if (128 + a.slots_bytes + static_cast<size_t>(stages) * a.stage_bytes > kSmemPerSm) return MOE_ERR_UNSUPPORTED;
    int per_sm = env_int("MOE_PERMUTE_CTAS_PER_SM", 48);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 64) per_sm = 64;
    int64_t grid = static_cast<int64_t>(moe_host::num_sms()) * per_sm;
    if (grid > a.n_groups) grid = a.n_groups;
    // no deeper ring than the groups a CTA gets: smaller CTAs, more of them resident
    const int64_t per_cta = (a.n_groups + grid - 1) / grid;
    if (per_cta < a.stages) {
        a.stages = static_cast<int>(per_cta < 2 ? 2 : per_cta);
        a.slots_bytes = slots_for(a.stages);
    }
    const size_t smem = 128 + a.slots_bytes + static_cast<size_t>(a.stages) * a.stage_bytes;
    if (cudaFuncSetAttribute(moe::permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemPerSm)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return moe_host::launch(moe::permute_kernel, dim3(static_cast<unsigned>(grid)), dim3(32), smem, stream, a);
}

namespace {
template <int KT, int U>
int launch_combine(const moe::CombineArgs& a, cudaStream_t stream) {
    const int warps_per_block = moe::COMBINE_THREADS / 32;
    int64_t blocks = (static_cast<int64_t>(a.N) + warps_per_block - 1) / warps_per_block;
    const int64_t cap = static_cast<int64_t>(moe_host::num_sms()) * env_int("MOE_COMBINE_BLOCKS_PER_SM", 8);
    if (blocks > cap) blocks = cap;
    return moe_host::launch(moe::combine_kernel<KT, U>, dim3(static_cast<unsigned>(blocks)),
                            dim3(moe::COMBINE_THREADS), 0, stream, a);
}
}  // namespace

extern "C" MOE_API int moe_combine(const uint16_t* y, const float* topk_w, int N, int K, int H, int E,
                                   int alignment, const MoePlanOut* plan, uint16_t* out, cudaStream_t stream) {
    // N = 0 (an empty batch): no output rows; the N-sized arrays may be null
    if (plan == nullptr || plan->status == nullptr ||
        (N > 0 && (y == nullptr || topk_w == nullptr || out == nullptr || plan->dst == nullptr)))
        return MOE_ERR_INVALID_ARG;
    if (N < 0 || K < 1 || K > 32 || E < 1 || E > 1024 || K > E || alignment < 1 || H < 8 || H % 8 != 0)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(topk_w, 4) || !aligned(plan->dst, 4))
        return MOE_ERR_INVALID_ARG;
    const int64_t p_cap = moe_plan_capacity_rows(N, E, K, alignment);
    if (p_cap < 0 || p_cap >= (int64_t(1) << 31) - 1) return MOE_ERR_INVALID_ARG;
    if (N == 0) return MOE_OK;
    moe::CombineArgs a;
    a.y = y;
    a.w = topk_w;
    a.dst = plan->dst;
    a.out = out;
    a.status = plan->status;
    a.N = N;
    a.K = K;
    a.H = H;
    a.p_cap = p_cap;
    switch (K) {
        case 1: return launch_combine<1, 8>(a, stream);
        case 2: return launch_combine<2, 8>(a, stream);
        case 4: return launch_combine<4, 4>(a, stream);
        case 6: return launch_combine<6, 2>(a, stream);
        case 8: return launch_combine<8, 2>(a, stream);
        default: return launch_combine<0, 1>(a, stream);
    }
}
