// balance.cu -- capacity-balanced logical-rank plan with redundant experts
// (MoonEP moonep/planning.py, PlanningKernel: the rank-0 balancing matrix z,
// the per-owner allocation of expert pairs to other ranks, the top-B remote
// expert selection, per-rank padded groups, and the dst computation by the
// allocation prefix with the rank * NvS + loff encoding), in its one-GPU
// form: a single source rank, so the prefix over source ranks of tokens per
// expert is the plain plan's count.
//
// Launch 1 (balance_kernel), one CTA of 32 warps, in order:
//   - warp 0: while some rank is above CAP and some below, move the largest
//     shortfall from the largest surplus (ties: lower rank); each step zeroes
//     one rank and a zeroed rank never moves again, so at most R steps;
//   - one warp per owner rank: hand the owner's expert pairs to its quota
//     ranks, largest quota and largest remaining expert first (ties: lower
//     index), then alloc_cumsum by a warp scan per expert.
//   alloc stays in shared memory when R * (E + 1) is small enough (the large
//   workload's 64 x 257 is).
// Launch 2 (balance_groups_kernel), a warp per destination rank: count its
//   remote experts, pick the top B by pairs (ties to the larger expert
//   index, -1 once no pairs remain), then a warp scan over its E + B groups
//   for the padded cu_seqlens, zero-fill ranges and expert offsets.
// Launch 3 (balance_dst_kernel), a lane per pair: each pair's position
//   among its expert's pairs comes from the plain plan (slot - cu[e]); a
//   binary search over alloc_cumsum finds its rank; duplicates by rank as in
//   MoonEP's canonicalisation.
#include "moe_common.cuh"

namespace moe {

constexpr int BAL_THREADS = 1024;
constexpr int BAL_WARPS = BAL_THREADS / 32;
constexpr int BAL_MAX_B = 64;

struct BalanceArgs {
    const int32_t* topk;
    const int32_t* counts;     // plain plan tokens_per_expert [E]
    const int32_t* cu;         // plain plan cu_seqlens [E+1]
    const int32_t* plain_dst;  // plain plan dst [N*K]
    int32_t* status;           // plain plan status
    MoeBalancedPlanOut out;
    int N, E, K, R, epn, tp, B;
    int32_t cap, NvS;
    int alloc_in_smem;  // balance_kernel keeps alloc [R][E] in shared memory
};

// Largest value, lowest index among equals, across the warp (idx >= 0).
__device__ __forceinline__ void warp_argmax_low(int32_t& v, int32_t& idx) {
    const int32_t m = __reduce_max_sync(FULL_MASK, v);
    idx = static_cast<int32_t>(__reduce_min_sync(FULL_MASK, v == m ? static_cast<uint32_t>(idx) : 0xffffffffu));
    v = m;
}
// Smallest value, lowest index among equals.
__device__ __forceinline__ void warp_argmin_low(int32_t& v, int32_t& idx) {
    const int32_t m = __reduce_min_sync(FULL_MASK, v);
    idx = static_cast<int32_t>(__reduce_min_sync(FULL_MASK, v == m ? static_cast<uint32_t>(idx) : 0xffffffffu));
    v = m;
}

__global__ void __launch_bounds__(BAL_THREADS) balance_kernel(const BalanceArgs a) {
    extern __shared__ __align__(16) int32_t s_dyn[];
    const int E = a.E, R = a.R, B = a.B, epn = a.epn;
    int32_t* s_z = s_dyn;                      // [R][R]
    int32_t* s_bal = s_z + R * R;              // [R]
    int32_t* s_rem = s_bal + R;                // [E] remaining pairs per expert
    int32_t* s_q = s_rem + E;                  // [BAL_WARPS][R] quotas
    int32_t* s_pick = s_q + BAL_WARPS * R;     // [BAL_WARPS][BAL_MAX_B]
    // alloc [R][E]: in shared memory when it fits (rows padded to E + 1 so a
    // column read is conflict-free; copied out at the end), else the output
    // itself; A is a generic pointer to either, AS its row stride
    int32_t* A = a.alloc_in_smem ? s_pick + BAL_WARPS * BAL_MAX_B : a.out.alloc;
    const int AS = a.alloc_in_smem ? E + 1 : E;
    __shared__ int s_bad;

    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_bad = ld_volatile_s32(a.status) != 0;
    __syncthreads();
    if (s_bad) return;

    // ---- zero the outputs written sparsely; load counts and balances
    for (int i = tid; i < R * R; i += BAL_THREADS) s_z[i] = 0;
    for (int i = tid; i < R * AS; i += BAL_THREADS) A[i] = 0;
    for (int i = tid; i < R * E; i += BAL_THREADS) a.out.expert_offsets[i] = 0;
    for (int i = tid; i < 2 * R; i += BAL_THREADS) a.out.remote_stats[i] = 0;
    for (int e = tid; e < E; e += BAL_THREADS) s_rem[e] = __ldg(a.counts + e);
    __syncthreads();
    for (int r = tid; r < R; r += BAL_THREADS) {
        int32_t g = 0;
        for (int e = r * epn; e < (r + 1) * epn; ++e) g += s_rem[e];
        s_bal[r] = g - a.cap;
    }
    __syncthreads();

    // ---- balancing (warp 0, balances in registers: rank lane + 32 q): at
    // most R steps
    if (warp == 0) {
        int32_t bv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) bv[q] = lane + 32 * q < R ? s_bal[lane + 32 * q] : 0;
        for (int step = 0; step <= R; ++step) {
            int32_t hv = INT32_MIN, hi = 0x7fffffff, lv = INT32_MAX, li = 0x7fffffff;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = lane + 32 * q;
                if (r < R) {
                    if (bv[q] > hv) {
                        hv = bv[q];
                        hi = r;
                    }
                    if (bv[q] < lv) {
                        lv = bv[q];
                        li = r;
                    }
                }
            }
            warp_argmax_low(hv, hi);
            warp_argmin_low(lv, li);
            if (hv <= 0 || lv >= 0) break;
            if (step == R) {  // cannot happen: each step zeroes a rank for good
                if (lane == 0) record_error(a.status, MOE_ERR_DEVICE_INDEX, -1);
                break;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (lane + 32 * q == hi) bv[q] += lv;
                if (lane + 32 * q == li) bv[q] = 0;
            }
            if (lane == 0) s_z[hi * R + li] = -lv;
        }
    }
    __syncthreads();

    // ---- allocation: a warp per owner rank
    for (int o = warp; o < R; o += BAL_WARPS) {
        int32_t* q = s_q + warp * R;
        for (int r = lane; r < R; r += 32) q[r] = s_z[o * R + r];
        __syncwarp();
        int32_t* rem = s_rem + o * epn;
        for (int it = 0; it <= R + epn; ++it) {  // each step exhausts a quota or an expert
            int32_t qv = INT32_MIN, qi = 0x7fffffff;
            for (int r = lane; r < R; r += 32)
                if (q[r] > qv) {
                    qv = q[r];
                    qi = r;
                }
            warp_argmax_low(qv, qi);
            if (qv <= 0) break;
            int32_t ev = INT32_MIN, ei = 0x7fffffff;
            for (int le = lane; le < epn; le += 32)
                if (rem[le] > ev) {
                    ev = rem[le];
                    ei = le;
                }
            warp_argmax_low(ev, ei);
            if (ev <= 0) break;
            const int32_t take = ev < qv ? ev : qv;
            if (lane == 0) {
                q[qi] = qv - take;
                rem[ei] = ev - take;
                A[static_cast<size_t>(qi) * AS + o * epn + ei] = take;
            }
            __syncwarp();
        }
        for (int le = lane; le < epn; le += 32) A[static_cast<size_t>(o) * AS + o * epn + le] = rem[le];
        __syncwarp();
    }
    __syncthreads();
    for (int i = tid; i < R * R; i += BAL_THREADS) a.out.z[i] = s_z[i];
    if (a.alloc_in_smem)
        for (int r = warp; r < R; r += BAL_WARPS)
            for (int e = lane; e < E; e += 32) a.out.alloc[static_cast<size_t>(r) * E + e] = A[static_cast<size_t>(r) * AS + e];
    // alloc_cumsum [E][R]: a warp per expert scans its column over the ranks
    // (row-contiguous stores)
    for (int e = warp; e < E; e += BAL_WARPS) {
        int32_t run = 0;
        for (int r0 = 0; r0 < R; r0 += 32) {
            const int r = r0 + lane;
            const int32_t v = r < R ? A[static_cast<size_t>(r) * AS + e] : 0;
            int32_t incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t y = __shfl_up_sync(FULL_MASK, incl, off);
                if (lane >= off) incl += y;
            }
            if (r < R) a.out.alloc_cumsum[static_cast<size_t>(e) * R + r] = run + incl;
            run += __shfl_sync(FULL_MASK, incl, 31);
        }
    }
}

// Launch 2 (balance_groups_kernel), a warp per destination rank: its remote
// experts, the top-B redundant experts by pairs (ties to the larger index,
// -1 once no pairs remain), then a warp scan over its E + B groups for the
// padded cu_seqlens, zero-fill ranges and expert offsets.
constexpr int BAL_GRP_WARPS = 8;

__global__ void __launch_bounds__(BAL_GRP_WARPS * 32) balance_groups_kernel(const BalanceArgs a) {
    __shared__ int32_t s_pick[BAL_GRP_WARPS][BAL_MAX_B];
    pdl_wait();
    pdl_trigger();
    if (ld_volatile_s32(a.status) != 0) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int E = a.E, R = a.R, B = a.B, epn = a.epn;
    const int d = blockIdx.x * BAL_GRP_WARPS + warp;
    if (d >= R) return;
    const int32_t* row = a.out.alloc + static_cast<size_t>(d) * E;
    uint32_t cleared = 0u, picked = 0u;  // bit j: expert lane + 32 j (E <= 1024)
    int nremote = 0;
    for (int e = lane, j = 0; e < E; e += 32, ++j) {
        const bool local = e >= d * epn && e < (d + 1) * epn;
        nremote += (!local && __ldg(row + e) > 0) ? 1 : 0;
    }
    nremote = __reduce_add_sync(FULL_MASK, nremote);
    if (lane == 0) a.out.remote_stats[2 * d] = nremote;
    int32_t* picks = s_pick[warp];
    for (int slot = 0; slot < B; ++slot) {
        int32_t bv = 0, bi = -1;
        for (int e = lane, j = 0; e < E; e += 32, ++j) {
            const bool local = e >= d * epn && e < (d + 1) * epn;
            const int32_t c = (local || ((cleared >> j) & 1u)) ? 0 : __ldg(row + e);
            if (c >= bv) {  // ties to the larger index
                bv = c;
                bi = e;
            }
        }
        const int32_t m = __reduce_max_sync(FULL_MASK, bv);
        const int32_t best = static_cast<int32_t>(__reduce_max_sync(FULL_MASK, bv == m ? bi : -1));
        const int32_t pick = m > 0 ? best : -1;
        if (best >= 0 && (best & 31) == lane) {
            cleared |= 1u << (best >> 5);
            if (pick >= 0) picked |= 1u << (best >> 5);
        }
        if (lane == 0) {
            picks[slot] = pick;
            a.out.experts_to_copy[static_cast<size_t>(d) * B + slot] = pick;
            if (pick >= 0) atomicAdd(a.out.remote_stats + 2 * (pick / epn) + 1, 1);
        }
    }
    __syncwarp();
    int64_t run = 0;
    const int G = E + B;
    for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + lane;
        int32_t c = 0;
        int expert = -1;
        if (g < E) {
            if (!((picked >> (g0 >> 5)) & 1u)) {
                c = __ldg(row + g);
                expert = g;
            }
        } else if (g < G) {
            const int32_t sel = picks[g - E];
            if (sel >= 0) {
                c = __ldg(row + sel);
                expert = sel;
            }
        }
        const int64_t padded = c > 0 ? (static_cast<int64_t>(c) + a.tp - 1) / a.tp * a.tp : 0;
        int64_t incl = padded;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(FULL_MASK, incl, off);
            if (lane >= off) incl += y;
        }
        const int64_t base = run + incl - padded;
        if (g < G) {
            const size_t gi = static_cast<size_t>(d) * G + g;
            a.out.rank_cu_seqlens[gi] = static_cast<int32_t>(base + padded);
            const bool pad = c > 0 && padded > c;
            a.out.rank_zero_fill[2 * gi] = pad ? static_cast<int32_t>(base + c) : 0;
            a.out.rank_zero_fill[2 * gi + 1] = pad ? static_cast<int32_t>(padded - c) : 0;
            if (c > 0) a.out.expert_offsets[static_cast<size_t>(d) * E + expert] = static_cast<int32_t>(base);
        }
        run += __shfl_sync(FULL_MASK, incl, 31);
    }
    if (lane == 0 && run > a.NvS) record_error(a.status, MOE_ERR_DEVICE_CAPACITY, d);
}

constexpr int BAL_DST_THREADS = 256;

// A lane per pair: 32 / K tokens per warp, lane (token, k) in k order.  The
// pair's position among its expert's pairs is slot - cu[e] from the plain
// plan; the first rank whose allocation prefix exceeds it is its rank; a
// later k of the same token on the same rank is a duplicate (match.any on
// (token, rank), the lowest lane is the primary).
__global__ void __launch_bounds__(BAL_DST_THREADS) balance_dst_kernel(const BalanceArgs a) {
    pdl_wait();
    pdl_trigger();
    if (ld_volatile_s32(a.status) != 0) return;
    const int lane = threadIdx.x & 31;
    const int E = a.E, K = a.K, R = a.R;
    const int tpw = 32 / K;
    const int tok_in = lane / K, k = lane - tok_in * K;
    const int64_t gwarp = (static_cast<int64_t>(blockIdx.x) * BAL_DST_THREADS + threadIdx.x) >> 5;
    const int64_t s = gwarp * tpw + tok_in;
    bool ok = tok_in < tpw && s < a.N;
    const int64_t f = s * K + k;
    int lo = 0;
    int32_t d = 0;
    if (ok) {
        const int e = __ldg(a.topk + f);
        if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
            record_error(a.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(f));
            ok = false;
        } else {
            const int32_t gr = raw_slot(__ldg(a.plain_dst + f)) - __ldg(a.cu + e);
            const int32_t* ac = a.out.alloc_cumsum + static_cast<size_t>(e) * R;
            int hi = R;  // first rank whose prefix exceeds gr
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(ac + mid) > gr)
                    hi = mid;
                else
                    lo = mid + 1;
            }
            if (lo >= R || gr < 0) {
                record_error(a.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(f));
                ok = false;
            } else {
                const int32_t pc = lo > 0 ? __ldg(ac + lo - 1) : 0;
                d = lo * a.NvS + __ldg(a.out.expert_offsets + static_cast<size_t>(lo) * E + e) + (gr - pc);
            }
        }
    }
    const unsigned peers = __match_any_sync(FULL_MASK, ok ? static_cast<unsigned>(tok_in * 128 + lo) : 0xffffffffu);
    if (ok) a.out.dst[f] = (peers & ((1u << lane) - 1u)) ? -d - 1 : d;
}

}  // namespace moe

// ---------------------------------------------------------------- host
namespace {
bool aligned4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % 4) == 0; }
}  // namespace

extern "C" MOE_API int moe_plan_balanced(const MoePlanOut* plan, const int32_t* topk_idx, int N, int E, int K,
                                         int R, int token_padding, int32_t capacity, int B, int32_t NvS,
                                         const MoeBalancedPlanOut* out, cudaStream_t stream) {
    // N = 0 (an empty batch) is valid: no pairs to balance, every output
    // matrix zero and no redundant expert; topk_idx and the dst arrays have
    // no elements and may be null
    if (plan == nullptr || out == nullptr || (N > 0 && topk_idx == nullptr)) return MOE_ERR_INVALID_ARG;
    if (N < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E || R < 1 || R > 128 || E % R != 0)
        return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(N) * K >= (int64_t(1) << 30)) return MOE_ERR_INVALID_ARG;
    if (token_padding < 1 || B < 0 || B > moe::BAL_MAX_B || NvS < 1 || capacity < 0) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(R) * NvS >= (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
    const void* in[] = {plan->tokens_per_expert, plan->cu_seqlens, plan->status};
    for (const void* p : in)
        if (!aligned4(p)) return MOE_ERR_INVALID_ARG;
    if (N > 0 && (!aligned4(plan->dst) || !aligned4(topk_idx) || !aligned4(out->dst))) return MOE_ERR_INVALID_ARG;
    const void* outs[] = {out->z, out->alloc, out->alloc_cumsum, out->remote_stats, out->rank_cu_seqlens,
                          out->rank_zero_fill, out->expert_offsets};
    for (const void* p : outs)
        if (!aligned4(p)) return MOE_ERR_INVALID_ARG;
    if (B > 0 && !aligned4(out->experts_to_copy)) return MOE_ERR_INVALID_ARG;

    moe::BalanceArgs a;
    a.topk = topk_idx;
    a.counts = plan->tokens_per_expert;
    a.cu = plan->cu_seqlens;
    a.plain_dst = plan->dst;
    a.status = plan->status;
    a.out = *out;
    a.N = N;
    a.E = E;
    a.K = K;
    a.R = R;
    a.epn = E / R;
    a.tp = token_padding;
    a.B = B;
    a.cap = capacity;
    a.NvS = NvS;
    size_t smem = sizeof(int32_t) * (static_cast<size_t>(R) * R + R + E + static_cast<size_t>(moe::BAL_WARPS) * R +
                                     static_cast<size_t>(moe::BAL_WARPS) * moe::BAL_MAX_B);
    const size_t alloc_bytes = sizeof(int32_t) * static_cast<size_t>(R) * (E + 1);
    a.alloc_in_smem = smem + alloc_bytes <= 200 * 1024 ? 1 : 0;
    if (a.alloc_in_smem) smem += alloc_bytes;
    if (cudaFuncSetAttribute(moe::balance_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return MOE_ERR_CUDA;
    int rc = moe_host::launch(moe::balance_kernel, dim3(1), dim3(moe::BAL_THREADS), smem, stream, a);
    if (rc != MOE_OK) return rc;
    rc = moe_host::launch(moe::balance_groups_kernel, dim3((R + moe::BAL_GRP_WARPS - 1) / moe::BAL_GRP_WARPS),
                          dim3(moe::BAL_GRP_WARPS * 32), 0, stream, a);
    if (rc != MOE_OK) return rc;
    if (N == 0) return MOE_OK;  // no pairs: no dst to write
    const int64_t warps = (static_cast<int64_t>(N) + 32 / K - 1) / (32 / K);
    const unsigned blocks = static_cast<unsigned>((warps * 32 + moe::BAL_DST_THREADS - 1) / moe::BAL_DST_THREADS);
    return moe_host::launch(moe::balance_dst_kernel, dim3(blocks), dim3(moe::BAL_DST_THREADS), 0, stream, a);
}
