// plan.cu -- dispatch plan for one GPU (sm_103a): histogram, aligned
// offsets, stable slots, per-rank duplicate detection, rank matrices and
// the dedup structures.  Four paths compute the identical plan:
//   - plan_small_kernel (default for E <= 32, R <= 32): one cluster launch,
//     lanes own experts and ranks, counts pushed between CTAs (described
//     at the kernel);
//   - plan_count_kernel + plan_scatter_kernel (default otherwise): two
//     launches with a decoupled look-back, described below;
//   - plan_cluster_kernel and plan_grid_kernel: one launch for any E, on
//     request (MOE_PLAN_PATH), described at the kernels.
//
// Pairs are cut into tiles of whole tokens.  Inside a tile each warp owns a
// contiguous run of tokens and walks it in iterations of floor(32/K) tokens,
// one lane per (token, k) pair, so lanes are in flat-pair order.
//
// Launch 1 (plan_count_kernel), one CTA per tile, tile id from a ticket so
// that a CTA only ever waits on tiles already running:
//   - per-tile counts of every "column": the E experts, then tokens per rank
//     (R columns), then (groups, duplicates);  __match_any_sync groups lanes
//     with the same expert so one leader adds the run length (MoonEP
//     moonep/planning.py, run_c1 pass A), and groups lanes with the same
//     (token, rank) for the duplicate test;
//   - a decoupled look-back per column gives the exclusive prefix over
//     earlier tiles (the single-pass replacement of MoonEP's grid-wide
//     per-expert prefix over blocks and of TensorRT-LLM's atomic tile
//     offsets); flags carry a call epoch so nothing needs clearing, waits
//     are bounded in time;
//   - the last tile holds the totals and writes tokens_per_expert, the
//     alignment-padded cu_seqlens and zero_fill_ranges (MoonEP per-rank
//     cu_seqlens / zero_fill_ranges; DeepEP notify_dispatch aligned counts)
//     and the rank arrays (DeepEP notify_dispatch rank prefix).
// Launch 2 (plan_scatter_kernel), one CTA per tile:
//   - re-derives each pair's rank among same-expert pairs of its warp run
//     (match.any + popc, per-warp running counts in shared memory), scans
//     the runs per expert, and writes the canonical slot
//     cu[e] + (pairs of e in earlier tiles) + (in earlier runs) + rank;
//   - dst = slot for the first pair of a token on a rank, -slot-1 for the
//     later ones (MoonEP duplicate canonicalisation), src_of_slot (MoonEP
//     src_info), is_token_in_rank, and the dedup structures in (token,
//     first k) order;
//   - -1 into the padding rows and unused capacity of src_of_slot.
#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "moe_common.cuh"
#include "route_core.cuh"

namespace moe {

constexpr int PLAN_THREADS = 1024;
constexpr int PLAN_WARPS = PLAN_THREADS / 32;
constexpr int PLAN_IPT_MAX = 8;
constexpr int LOOKBACK_WINDOW = 16;
constexpr uint32_t ST_AGG = 1u, ST_PRE = 2u, ST_ERR = 3u;

struct WsHeader {
    uint32_t epoch;   // epoch of the last completed call
    uint32_t ticket;  // next tile id of the running call
    uint32_t done;    // CTAs of the running call that finished
    uint32_t pad[13];
};
static_assert(sizeof(WsHeader) == 64, "header size");

struct PlanArgs {
    const int32_t* topk;
    MoePlanOut out;
    WsHeader* hdr;
    uint64_t* flags;       // [T][C]
    int32_t* tile_prefix;  // [T][C]
    int N, E, K, R, epn, alignment;
    uint64_t epn_magic;  // floor(2^32 / epn) + 1: e / epn == (e * epn_magic) >> 32 for e < 2048
    int tpw, ipt, tile_tokens, T, C;
    int64_t p_cap;
    int skip_tile;
    int64_t timeout_ns;
};

// A flag word: tag in the high half, state and value in the low half.  The
// tag is the call epoch with bit 31 set: counts and prefixes left in the
// workspace by calls of other sizes are below 2^30, so no leftover word can
// carry the tag of the running call.
__device__ __forceinline__ uint32_t flag_tag(uint32_t epoch) { return epoch | 0x80000000u; }
// Rank of expert e (e < 2048) without an integer division.
__device__ __forceinline__ int rank_of(const PlanArgs& a, int e) {
    return static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(e)) * a.epn_magic) >> 32);
}

// First 16-byte boundary at or after p, measured from the start of the
// dynamic shared memory block (the tile's is_token_in_rank bytes are copied
// out with 16-byte vectors).
__device__ __forceinline__ uint8_t* align16_after(int32_t* base, int32_t* p) {
    const ptrdiff_t ints = p - base;
    return reinterpret_cast<uint8_t*>(base + ((ints + 3) & ~static_cast<ptrdiff_t>(3)));
}

__device__ __forceinline__ uint64_t pack_flag(uint32_t epoch, uint32_t st, uint32_t v) {
    return (static_cast<uint64_t>(flag_tag(epoch)) << 32) | (static_cast<uint64_t>(st) << 30) | (v & 0x3fffffffu);
}

// Exclusive prefix sum of n values in shared memory by one CTA of WARPS
// warps: out[0] = 0, out[i+1] = out[i] + in[i].  `in` and `out` may not
// alias; s_warp holds WARPS + 1 ints.
template <int WARPS>
__device__ void block_exclusive_scan(const int32_t* in, int n, int32_t* out, int32_t* s_warp) {
    constexpr int THREADS = WARPS * 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = (n + THREADS - 1) / THREADS;
    const int b = min(n, tid * chunk), e = min(n, b + chunk);
    int32_t local = 0;
    for (int i = b; i < e; ++i) local += in[i];
    int32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(FULL_MASK, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {  // exclusive scan of the warp totals
        const int32_t v = lane < WARPS ? s_warp[lane] : 0;
        int32_t w_incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(FULL_MASK, w_incl, off);
            if (lane >= off) w_incl += y;
        }
        if (lane < WARPS) s_warp[lane] = w_incl - v;
        if (lane == WARPS - 1) s_warp[WARPS] = w_incl;
    }
    __syncthreads();
    int32_t run = s_warp[warp] + incl - local;
    for (int i = b; i < e; ++i) {
        out[i] = run;
        run += in[i];
    }
    if (tid == 0) out[n] = s_warp[WARPS];
    __syncthreads();
}

// ---------------------------------------------------------------- shared pieces
// From the column totals s_tot (E expert counts, R per-rank token counts,
// groups, duplicates): cu_seqlens into s_cu[0..E] for the calling CTA and,
// when `write`, every totals-derived output (MoonEP per-rank cu_seqlens and
// zero_fill_ranges with padded = round_up(count, alignment) for count > 0;
// DeepEP notify_dispatch rank prefix).  s_pad: E + R + 2 ints of scratch.
// Contains __syncthreads: every thread of the CTA (WARPS warps) calls it.
template <int WARPS>
__device__ void plan_totals(const PlanArgs& a, const int32_t* s_tot, int32_t* s_pad, int32_t* s_cu, int32_t* s_warp,
                            bool write) {
    constexpr int THREADS = WARPS * 32;
    const int tid = threadIdx.x;
    const int E = a.E, R = a.R, al = a.alignment;
    for (int e = tid; e < E; e += THREADS) {
        const int32_t c = s_tot[e];
        s_pad[e] = c > 0 ? static_cast<int32_t>((static_cast<int64_t>(c) + al - 1) / al * al) : 0;
    }
    __syncthreads();
    block_exclusive_scan<WARPS>(s_pad, E, s_cu, s_warp);  // s_cu[0..E] = cu
    if (!write) return;
    for (int e = tid; e < E; e += THREADS) {
        a.out.tokens_per_expert[e] = s_tot[e];
        const int32_t pad = s_pad[e] - s_tot[e];
        a.out.zero_fill_ranges[2 * e] = pad > 0 ? s_cu[e] + s_tot[e] : 0;
        a.out.zero_fill_ranges[2 * e + 1] = pad > 0 ? pad : 0;
    }
    for (int e = tid; e <= E; e += THREADS) a.out.cu_seqlens[e] = s_cu[e];
    for (int r = tid; r <= R; r += THREADS) a.out.rank_slot_offsets[r] = s_cu[r * a.epn];
    for (int r = tid; r < R; r += THREADS) {
        int32_t pairs = 0;
        for (int e = r * a.epn; e < (r + 1) * a.epn; ++e) pairs += s_tot[e];
        a.out.pairs_per_rank[r] = pairs;
        a.out.tokens_per_rank[r] = s_tot[E + r];
    }
    if (tid == 0) {
        a.out.dup_counts[0] = s_tot[E + R];
        a.out.dup_counts[1] = s_tot[E + R + 1];
    }
    __syncthreads();
    block_exclusive_scan<WARPS>(s_tot + E, R, s_pad, s_warp);  // s_pad[0..R] = rank prefix
    for (int r = tid; r <= R; r += THREADS) a.out.rank_prefix[r] = s_pad[r];
}

// Per-pair results of a tile's first pass, kept in shared memory (8 bytes
// per pair, s_items[warp][step][lane]) until the slots are known, so the
// item loops stay rolled and the kernels' code stays small (they run once
// per SM, with a cold instruction cache).
//   x: expert (11 bits, 0x7ff = inactive lane) | rank among the same
//      expert's pairs of the warp run (10 bits) | duplicate (1) | opens a
//      group (1) | duplicates in the group (5)
//   y: group index (opener) or duplicate position (16) | first duplicate
//      position of the group (16), both within the warp run
__device__ __forceinline__ uint2 pack_item(int e, int rank, bool dup, bool opens, int ndup, int ia, int ib) {
    return make_uint2(static_cast<uint32_t>(e) | (static_cast<uint32_t>(rank) << 11) | (dup ? 1u << 21 : 0u) |
                          (opens ? 1u << 22 : 0u) | (static_cast<uint32_t>(ndup) << 23),
                      static_cast<uint32_t>(ia) | (static_cast<uint32_t>(ib) << 16));
}
constexpr uint32_t ITEM_NONE = 0x7ffu;

// First pass over a tile: per-warp running counts of every expert (s_wc,
// [PLAN_WARPS][E], zeroed), each pair's rank among the same expert's pairs
// of its warp run (match.any + popc: lanes are in flat-pair order), the
// duplicate test per (token, rank) (match.any on the pair's token and rank),
// group / duplicate positions within the warp run (ballots), the tile's
// is_token_in_rank rows (s_itr, zeroed) and per-warp group / duplicate
// totals (s_wg, s_wd).  With s_rtok non-null it also counts the tile's
// tokens per rank.  Reads only topk_idx.
__device__ __noinline__ void tile_phase1(const PlanArgs& a, int tile, int32_t* s_wc, uint8_t* s_itr, int32_t* s_wg,
                                         int32_t* s_wd, int32_t* s_rtok, uint2* s_items) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, K = a.K, R = a.R;
    const int64_t tok0 = static_cast<int64_t>(tile) * a.tile_tokens;
    const unsigned lt = (1u << lane) - 1u;
    const int act = a.tpw * K;
    const int tok_in_iter = lane / K, k = lane - (lane / K) * K;
    const int tok_lane0 = tok_in_iter * K;
    const unsigned below_tok = (1u << tok_lane0) - 1u;
    const unsigned tokmask = (K == 32 ? FULL_MASK : ((1u << K) - 1u)) << tok_lane0;  // this token's lanes
    const int rbits = R > 1 ? 32 - __clz(R - 1) : 0;
    const int ebits = E > 1 ? 32 - __clz(E - 1) : 0;
    // all of this lane's expert ids first: one memory latency for the tile
    int ids[PLAN_IPT_MAX];
#pragma unroll
    for (int i = 0; i < PLAN_IPT_MAX; ++i) {
        const int64_t s = tok0 + static_cast<int64_t>(warp * a.ipt + i) * a.tpw + tok_in_iter;
        ids[i] = (i < a.ipt && lane < act && s < a.N) ? __ldg(a.topk + s * K + k) : -1;
    }
    int run_g = 0, run_d = 0;
#pragma unroll 1
    for (int i = 0; i < a.ipt; ++i) {
        int id = ids[0];
#pragma unroll
        for (int q = 1; q < PLAN_IPT_MAX; ++q)
            if (q == i) id = ids[q];
        const int64_t s = tok0 + static_cast<int64_t>(warp * a.ipt + i) * a.tpw + tok_in_iter;
        bool active = lane < act && s < a.N;
        int e = E;
        if (active) {
            e = id;
            if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(s * K + k));
                active = false;
                e = E;
            }
        }
        // lanes with the same expert: one ballot per bit of the expert id
        // (these passes are latency-bound; a match.any is a long wait)
        const unsigned amask = __ballot_sync(FULL_MASK, active);
        unsigned pe = amask;
        for (int b = 0; b < ebits; ++b) {
            const unsigned eb = __ballot_sync(FULL_MASK, (e >> b) & 1);
            pe &= ((e >> b) & 1) ? eb : ~eb;
        }
        const unsigned peers = active ? pe : (1u << lane);
        const int base = active ? s_wc[warp * E + e] : 0;
        const int wr = base + __popc(peers & lt);
        __syncwarp();
        if (active && (peers & lt) == 0u) s_wc[warp * E + e] = base + __popc(peers);
        __syncwarp();

        const int r = active ? rank_of(a, e) : 0;
        // lanes on the same rank: one ballot per bit of the rank (cheaper
        // than a match.any on a (token, rank) key); pd = this token's pairs
        // on this lane's rank
        unsigned pr = amask;
        for (int b = 0; b < rbits; ++b) {
            const unsigned rb = __ballot_sync(FULL_MASK, (r >> b) & 1);
            pr &= ((r >> b) & 1) ? rb : ~rb;
        }
        const unsigned pd = active ? (pr & tokmask) : (1u << lane);
        const bool prim = active && (pd & lt) == 0u;
        const bool dup = active && !prim;
        const bool opens = prim && __popc(pd) >= 2;
        const unsigned gball = __ballot_sync(FULL_MASK, opens);
        const unsigned dball = __ballot_sync(FULL_MASK, dup);
        // Duplicates of a token are laid out group after group (groups in
        // order of their primary lane = first k), k order inside a group.
        // A warp scan of the group sizes gives the duplicates of the
        // token's groups that open before a given lane.
        const int my_p = __ffs(pd) - 1;
        const int gsz = opens ? __popc(pd) - 1 : 0;
        int incl = gsz;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(FULL_MASK, incl, off);
            if (lane >= off) incl += y;
        }
        const int excl = incl - gsz;
        const int tok_base = __shfl_sync(FULL_MASK, excl, tok_lane0);
        const int groups_before = __shfl_sync(FULL_MASK, excl, my_p) - tok_base;
        const int before = groups_before + (dup ? __popc(pd & lt) - 1 : 0);
        const int dup_pos = run_d + __popc(dball & below_tok) + before;
        if (prim) s_itr[(s - tok0) * R + r] = 1;
        if (s_rtok != nullptr) {
            // tokens per rank: one add per distinct rank of the warp step
            // (per-lane adds on R counters serialise)
            const unsigned same = pr & __ballot_sync(FULL_MASK, prim);
            if (prim && (same & lt) == 0u) atomicAdd(&s_rtok[r], __popc(same));
        }
        s_items[(warp * a.ipt + i) * 32 + lane] =
            active ? pack_item(e, wr, dup, opens, __popc(pd) - 1, opens ? run_g + __popc(gball & lt) : dup_pos, dup_pos)
                   : make_uint2(ITEM_NONE, 0u);
        run_g += __popc(gball);
        run_d += __popc(dball);
    }
    if (lane == 0) {
        s_wg[warp] = run_g;
        s_wd[warp] = run_d;
    }
}

// Exclusive scan of the per-warp-run values by one warp (lane w holds warp
// run w's value), written back with `base` added.
template <int WARPS>
__device__ __forceinline__ void warp_scan_runs(int32_t* s_val, int32_t base) {
    const int lane = threadIdx.x & 31;
    int32_t v = lane < WARPS ? s_val[lane] : 0;
    int32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(FULL_MASK, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane < WARPS) s_val[lane] = base + incl - v;
}

// Second pass over a tile, after the bases are known: s_base[e] = first slot
// of expert e in this tile, g_base / d_base = groups / duplicates of earlier
// tiles.  Turns the per-warp counts into per-warp bases, then writes dst,
// src_of_slot, dup_groups, dup_loffs and the tile's is_token_in_rank rows.
template <int WARPS>
__device__ __noinline__ void tile_phase3(const PlanArgs& a, int tile, const int32_t* s_base, int32_t g_base,
                                         int32_t d_base, int32_t* s_wc, int32_t* s_wg, int32_t* s_wd,
                                         const uint8_t* s_itr, const uint2* s_items) {
    constexpr int THREADS = WARPS * 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, K = a.K, R = a.R;
    const int64_t tok0 = static_cast<int64_t>(tile) * a.tile_tokens;
    // per (warp run, expert): the expert's pairs in earlier warp runs; a
    // thread per expert (neighbouring threads, neighbouring banks), all its
    // loads issued before the running sum
    for (int e = tid; e < E; e += THREADS) {
        int32_t v[WARPS];
#pragma unroll
        for (int w = 0; w < WARPS; ++w) v[w] = s_wc[w * E + e];
        int32_t run = s_base[e];
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            s_wc[w * E + e] = run;
            run += v[w];
        }
    }
    if (warp == WARPS - 1) warp_scan_runs<WARPS>(s_wg, g_base);
    if (warp == WARPS - 2) warp_scan_runs<WARPS>(s_wd, d_base);
    __syncthreads();

    const int tok_in_iter = lane / K, k = lane - (lane / K) * K;
    const int32_t wg = s_wg[warp], wd = s_wd[warp];
#pragma unroll 1
    for (int i = 0; i < a.ipt; ++i) {
        const uint2 it = s_items[(warp * a.ipt + i) * 32 + lane];
        const uint32_t e = it.x & 0x7ffu;
        if (e == ITEM_NONE) continue;
        const int64_t s = tok0 + static_cast<int64_t>(warp * a.ipt + i) * a.tpw + tok_in_iter;
        const int64_t f = s * K + k;
        const int32_t slot = s_wc[warp * E + e] + static_cast<int32_t>((it.x >> 11) & 0x3ffu);
        if (slot < 0 || static_cast<int64_t>(slot) >= a.p_cap) {
            record_error(a.out.status, MOE_ERR_DEVICE_INDEX, slot);
            continue;
        }
        const bool dup = (it.x >> 21) & 1u;
        const bool opens = (it.x >> 22) & 1u;
        const int32_t ia = static_cast<int32_t>(it.y & 0xffffu), ib = static_cast<int32_t>(it.y >> 16);
        a.out.dst[f] = dup ? -slot - 1 : slot;
        a.out.src_of_slot[slot] = static_cast<int32_t>(f);
        if (opens) {
            const int64_t g = static_cast<int64_t>(wg) + ia;
            if (g >= static_cast<int64_t>(a.N) * (K / 2)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(g));
                continue;
            }
            int32_t* row = a.out.dup_groups + 3 * g;
            row[0] = slot;
            row[1] = wd + ib;
            row[2] = static_cast<int32_t>(it.x >> 23);
        } else if (dup) {
            const int64_t pos = static_cast<int64_t>(wd) + ia;
            if (pos >= static_cast<int64_t>(a.N) * (K - 1)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(pos));
                continue;
            }
            a.out.dup_loffs[pos] = slot;
        }
    }

    // is_token_in_rank rows of this tile (16-byte stores when aligned)
    const int64_t ntok = min(static_cast<int64_t>(a.tile_tokens), static_cast<int64_t>(a.N) - tok0);
    const int64_t nbytes = ntok * R;
    uint8_t* g = a.out.is_token_in_rank + tok0 * R;
    if ((reinterpret_cast<uintptr_t>(g) & 15u) == 0) {
        const int64_t nvec = nbytes / 16;
        for (int64_t v = tid; v < nvec; v += THREADS)
            reinterpret_cast<uint4*>(g)[v] = reinterpret_cast<const uint4*>(s_itr)[v];
        for (int64_t b = nvec * 16 + tid; b < nbytes; b += THREADS) g[b] = s_itr[b];
    } else {
        for (int64_t b = tid; b < nbytes; b += THREADS) g[b] = s_itr[b];
    }
}

// -1 into src_of_slot for the padding rows of experts tile, tile + T, ...
// (cu, cnt: cu_seqlens and per-expert counts) and for this tile's share of
// the unused rows [P, P_cap).
template <int WARPS>
__device__ __forceinline__ void fill_unused(const PlanArgs& a, int tile, int T, const int32_t* cu, const int32_t* cnt) {
    constexpr int THREADS = WARPS * 32;
    const int tid = threadIdx.x;
    const int per = a.alignment - 1;  // at most this many padding rows per expert
    if (per > 0) {
        const int mine = (a.E - tile + T - 1) / T;  // experts tile, tile + T, ...
        for (int i = tid; i < mine * per; i += THREADS) {
            const int e = tile + (i / per) * T, j = i - (i / per) * per;
            const int32_t start = cu[e] + cnt[e];
            if (j < cu[e + 1] - start && start >= 0 && static_cast<int64_t>(start) + j < a.p_cap)
                a.out.src_of_slot[start + j] = -1;
        }
    }
    const int64_t P = cu[a.E];
    const int64_t rest = a.p_cap - P;
    const int64_t share = (rest + T - 1) / T;
    const int64_t b = P + share * tile, e = min(a.p_cap, b + share);
    for (int64_t j = b + tid; j < e; j += THREADS) a.out.src_of_slot[j] = -1;
}

// ---------------------------------------------------------------- launch 1
__global__ void __launch_bounds__(PLAN_THREADS) plan_count_kernel(const PlanArgs a) {
    extern __shared__ __align__(16) int32_t s_dyn[];
    int32_t* s_tot = s_dyn;               // [C]  counts, then totals
    int32_t* s_tmp = s_dyn + a.C;         // [E + R + 2] scratch for the last tile
    int32_t* s_scan = s_tmp + a.E + a.R + 2;  // [E + R + 2]
    __shared__ int32_t s_warp[PLAN_WARPS + 1];
    __shared__ int s_tile;
    __shared__ uint32_t s_epoch;
    __shared__ int s_err;

    pdl_wait();
    pdl_trigger();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, K = a.K, R = a.R, C = a.C;
    if (tid == 0) {
        s_tile = static_cast<int>(atomicAdd(&a.hdr->ticket, 1u));
        s_epoch = ((*reinterpret_cast<volatile uint32_t*>(&a.hdr->epoch) + 1u) & 0x7fffffffu);
        s_err = 0;
    }
    for (int c = tid; c < C; c += PLAN_THREADS) s_tot[c] = 0;
    __syncthreads();
    const int tile = s_tile;
    const uint32_t epoch = s_epoch;
    const bool tile_ok = tile >= 0 && tile < a.T;
    if (!tile_ok && tid == 0) record_error(a.out.status, MOE_ERR_WORKSPACE, tile);

    if (tile_ok) {
        // ---- per-tile counts
        const unsigned lt = (1u << lane) - 1u;
        const int act = a.tpw * K;
        const int tok_in_iter = lane / K, k = lane - (lane / K) * K;
        const unsigned tokmask = (K == 32 ? FULL_MASK : ((1u << K) - 1u)) << (tok_in_iter * K);
        const int rbits = R > 1 ? 32 - __clz(R - 1) : 0;
        const int ebits = E > 1 ? 32 - __clz(E - 1) : 0;
        const int64_t tok0 = static_cast<int64_t>(tile) * a.tile_tokens;
        // all of this lane's expert ids first: one memory latency for the tile
        int ids[PLAN_IPT_MAX];
#pragma unroll
        for (int i = 0; i < PLAN_IPT_MAX; ++i) {
            const int64_t s = tok0 + static_cast<int64_t>(warp * a.ipt + i) * a.tpw + tok_in_iter;
            ids[i] = (i < a.ipt && lane < act && s < a.N) ? __ldg(a.topk + s * K + k) : -1;
        }
        int my_groups = 0, my_dups = 0;
#pragma unroll 1
        for (int i = 0; i < a.ipt; ++i) {
            int id = ids[0];
#pragma unroll
            for (int q = 1; q < PLAN_IPT_MAX; ++q)
                if (q == i) id = ids[q];
            const int64_t s = tok0 + static_cast<int64_t>(warp * a.ipt + i) * a.tpw + tok_in_iter;
            bool active = lane < act && s < a.N;
            int e = E;
            if (active) {
                e = id;
                if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
                    record_error(a.out.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(s * K + k));
                    active = false;
                    e = E;
                }
            }
            // lanes with the same expert, then on the same rank: one ballot
            // per bit of the id
            const unsigned amask = __ballot_sync(FULL_MASK, active);
            unsigned peers = amask;
            for (int b = 0; b < ebits; ++b) {
                const unsigned eb = __ballot_sync(FULL_MASK, (e >> b) & 1);
                peers &= ((e >> b) & 1) ? eb : ~eb;
            }
            if (active && (peers & lt) == 0u) atomicAdd(&s_tot[e], __popc(peers));
            const int r = active ? rank_of(a, e) : 0;
            unsigned pr = amask;
            for (int b = 0; b < rbits; ++b) {
                const unsigned rb = __ballot_sync(FULL_MASK, (r >> b) & 1);
                pr &= ((r >> b) & 1) ? rb : ~rb;
            }
            const unsigned pd = pr & tokmask;  // this token's pairs on this lane's rank
            const bool prim = active && (pd & lt) == 0u;
            if (prim && __popc(pd) >= 2) ++my_groups;
            if (active && !prim) ++my_dups;
            const unsigned same = pr & __ballot_sync(FULL_MASK, prim);  // primaries on this rank
            if (prim && (same & lt) == 0u) atomicAdd(&s_tot[E + r], __popc(same));
        }
        my_groups = __reduce_add_sync(FULL_MASK, my_groups);
        my_dups = __reduce_add_sync(FULL_MASK, my_dups);
        if (lane == 0) {
            atomicAdd(&s_tot[E + R], my_groups);
            atomicAdd(&s_tot[E + R + 1], my_dups);
        }
        __syncthreads();

        // ---- decoupled look-back, one thread per column
        if (tile != a.skip_tile) {
            for (int c = tid; c < C; c += PLAN_THREADS) {
                const int32_t local = s_tot[c];
                uint64_t* mine = a.flags + static_cast<size_t>(tile) * C + c;
                int32_t excl = 0;
                bool err = false;
                if (tile == 0) {
                    st_relaxed_u64(mine, pack_flag(epoch, ST_PRE, static_cast<uint32_t>(local)));
                } else {
                    st_relaxed_u64(mine, pack_flag(epoch, ST_AGG, static_cast<uint32_t>(local)));
                    int j = tile - 1;
                    uint64_t t0 = 0;
                    while (true) {
                        uint64_t w[LOOKBACK_WINDOW];
#pragma unroll
                        for (int q = 0; q < LOOKBACK_WINDOW; ++q)
                            w[q] = (j - q >= 0) ? ld_relaxed_u64(a.flags + static_cast<size_t>(j - q) * C + c) : 0ull;
                        int consumed = 0;
                        bool done = false, stall = false;
#pragma unroll
                        for (int q = 0; q < LOOKBACK_WINDOW; ++q) {
                            if (done || stall) continue;
                            if (j - q < 0 || static_cast<uint32_t>(w[q] >> 32) != flag_tag(epoch)) {
                                stall = true;
                                continue;
                            }
                            const uint32_t st = static_cast<uint32_t>(w[q] >> 30) & 3u;
                            if (st == ST_ERR) {
                                err = true;
                                done = true;
                                continue;
                            }
                            excl += static_cast<int32_t>(w[q] & 0x3fffffffu);
                            ++consumed;
                            if (st == ST_PRE) done = true;
                        }
                        if (done) break;
                        j -= consumed;
                        if (stall) {
                            const uint64_t now = globaltimer_ns();
                            if (t0 == 0) {
                                t0 = now;
                            } else if (now - t0 > static_cast<uint64_t>(a.timeout_ns)) {
                                record_error(a.out.status, MOE_ERR_DEVICE_TIMEOUT, tile);
                                err = true;
                                break;
                            }
                            __nanosleep(100);
                        }
                    }
                    st_relaxed_u64(mine, err ? pack_flag(epoch, ST_ERR, 0u)
                                             : pack_flag(epoch, ST_PRE, static_cast<uint32_t>(excl + local)));
                }
                if (err) s_err = 1;
                a.tile_prefix[static_cast<size_t>(tile) * C + c] = excl;
                s_tot[c] = excl + local;
            }
        }
        __syncthreads();

        // ---- last tile: totals -> aligned offsets and rank arrays
        if (tile == a.T - 1 && tile != a.skip_tile && s_err == 0) plan_totals<PLAN_WARPS>(a, s_tot, s_tmp, s_scan, s_warp, true);
    }

    // ---- completion: the last CTA to finish closes the epoch
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&a.hdr->done, 1u);
        if (prev == gridDim.x - 1) {
            a.hdr->ticket = 0u;
            a.hdr->done = 0u;
            a.hdr->epoch = epoch;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------- launch 2
__global__ void __launch_bounds__(PLAN_THREADS) plan_scatter_kernel(const PlanArgs a) {
    extern __shared__ __align__(16) int32_t s_dyn[];
    uint2* s_items = reinterpret_cast<uint2*>(s_dyn);                  // [PLAN_WARPS][ipt][32]
    int32_t* s_wc = s_dyn + 2 * PLAN_WARPS * 32 * a.ipt;               // [PLAN_WARPS][E]
    int32_t* s_base = s_wc + PLAN_WARPS * a.E;                         // [E]
    uint8_t* s_itr = align16_after(s_dyn, s_base + a.E);               // [tile_tokens][R]
    __shared__ int32_t s_wg[PLAN_WARPS], s_wd[PLAN_WARPS];
    __shared__ int32_t s_bad;

    const int tid = threadIdx.x;
    const int E = a.E, R = a.R;
    const int tile = blockIdx.x;
    const int itr_bytes = a.tile_tokens * R;
    for (int i = tid; i < PLAN_WARPS * E; i += PLAN_THREADS) s_wc[i] = 0;
    for (int i = tid; i < (itr_bytes + 3) / 4; i += PLAN_THREADS) reinterpret_cast<int32_t*>(s_itr)[i] = 0;
    __syncthreads();

    // Reads only topk_idx, which was complete before launch 1 passed its wait.
    tile_phase1(a, tile, s_wc, s_itr, s_wg, s_wd, nullptr, s_items);

    // ---- everything below needs launch 1's outputs
    pdl_wait();
    pdl_trigger();
    if (tid == 0) s_bad = ld_volatile_s32(a.out.status) != 0 ? 1 : 0;
    __syncthreads();
    if (s_bad) return;
    const int32_t* tp = a.tile_prefix + static_cast<size_t>(tile) * a.C;
    for (int e = tid; e < E; e += PLAN_THREADS) s_base[e] = __ldg(a.out.cu_seqlens + e) + __ldg(tp + e);
    const int32_t g_base = __ldg(tp + E + R), d_base = __ldg(tp + E + R + 1);
    __syncthreads();
    tile_phase3<PLAN_WARPS>(a, tile, s_base, g_base, d_base, s_wc, s_wg, s_wd, s_itr, s_items);
    fill_unused<PLAN_WARPS>(a, tile, a.T, a.out.cu_seqlens, a.out.tokens_per_expert);
}

// ---------------------------------------------------------------- cluster path
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Address of `p` (this CTA's shared memory) in the shared memory of CTA
// `rank` of the cluster, then a load from it.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ int32_t ld_dsmem_s32(uint32_t addr) {
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// The whole plan in one launch for up to 16 tiles: one thread-block
// cluster, one CTA per tile.  Each CTA runs the tile's first pass, publishes
// its column counts in its own shared memory, and after a cluster barrier
// reads the other CTAs' counts through distributed shared memory: the sum
// over lower ranks is its exclusive prefix, the sum over all its totals.
// Every CTA scans the totals into cu_seqlens itself; rank 0 writes the
// totals-derived outputs.  No workspace, no look-back, no spin.
__global__ void __launch_bounds__(PLAN_THREADS) plan_cluster_kernel(const PlanArgs a) {
    extern __shared__ __align__(16) int32_t s_dyn[];
    const int E = a.E, R = a.R, C = a.C;
    uint2* s_items = reinterpret_cast<uint2*>(s_dyn);  // [PLAN_WARPS][ipt][32]
    int32_t* s_wc = s_dyn + 2 * PLAN_WARPS * 32 * a.ipt;  // [PLAN_WARPS][E]
    int32_t* s_cnt = s_wc + PLAN_WARPS * E;       // [C]  this tile's column counts
    int32_t* s_tot = s_cnt + C;                   // [C]  cluster totals
    int32_t* s_base = s_tot + C;                  // [E]
    int32_t* s_pad = s_base + E;                  // [E + R + 2]
    int32_t* s_cu = s_pad + E + R + 2;            // [E + R + 2]
    uint8_t* s_itr = align16_after(s_dyn, s_cu + E + R + 2);  // [tile_tokens][R]
    __shared__ int32_t s_wg[PLAN_WARPS], s_wd[PLAN_WARPS], s_warp[PLAN_WARPS + 1];
    __shared__ int32_t s_gd[2];

    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x;
    const uint32_t rank = cluster_ctarank();
    const uint32_t ncta = cluster_nctarank();
    const int tile = static_cast<int>(rank);
    const int itr_bytes = a.tile_tokens * R;
    for (int i = tid; i < PLAN_WARPS * E; i += PLAN_THREADS) s_wc[i] = 0;
    for (int i = tid; i < (itr_bytes + 3) / 4; i += PLAN_THREADS) reinterpret_cast<int32_t*>(s_itr)[i] = 0;
    for (int c = E + tid; c < C; c += PLAN_THREADS) s_cnt[c] = 0;
    __syncthreads();

    tile_phase1(a, tile, s_wc, s_itr, s_wg, s_wd, s_cnt + E, s_items);
    __syncthreads();
    for (int e = tid; e < E; e += PLAN_THREADS) {
        int32_t c = 0;
#pragma unroll
        for (int w = 0; w < PLAN_WARPS; ++w) c += s_wc[w * E + e];
        s_cnt[e] = c;
    }
    if ((tid >> 5) == 0) {
        const int lane = tid & 31;
        const int32_t g = __reduce_add_sync(FULL_MASK, lane < PLAN_WARPS ? s_wg[lane] : 0);
        const int32_t d = __reduce_add_sync(FULL_MASK, lane < PLAN_WARPS ? s_wd[lane] : 0);
        if (lane == 0) {
            s_cnt[E + R] = g;
            s_cnt[E + R + 1] = d;
        }
    }
    cluster_arrive();  // counts of every tile visible cluster-wide
    cluster_wait();

    for (int c = tid; c < C; c += PLAN_THREADS) {
        int32_t v[16];
#pragma unroll
        for (uint32_t q = 0; q < 16; ++q) v[q] = q < ncta ? ld_dsmem_s32(dsmem_addr(s_cnt + c, q)) : 0;
        int32_t excl = 0, tot = 0;
#pragma unroll
        for (uint32_t q = 0; q < 16; ++q) {
            if (q < rank) excl += v[q];
            tot += v[q];
        }
        s_tot[c] = tot;
        if (c < E) s_base[c] = excl;
        if (c == E + R) s_gd[0] = excl;
        if (c == E + R + 1) s_gd[1] = excl;
    }
    cluster_arrive();  // done reading the other CTAs' shared memory
    __syncthreads();

    plan_totals<PLAN_WARPS>(a, s_tot, s_pad, s_cu, s_warp, rank == 0);
    for (int e = tid; e < E; e += PLAN_THREADS) s_base[e] += s_cu[e];
    __syncthreads();
    tile_phase3<PLAN_WARPS>(a, tile, s_base, s_gd[0], s_gd[1], s_wc, s_wg, s_wd, s_itr, s_items);
    fill_unused<PLAN_WARPS>(a, tile, static_cast<int>(ncta), s_cu, s_tot);
    cluster_wait();  // keep this CTA's shared memory alive until all reads are done
}

// ---------------------------------------------------------------- small-E path
// E <= 32 and R <= 32 (NB = 3 bits for E, R <= 8, else 5): one
// thread-block cluster of T <= 16 CTAs of 32 warps, IPT warp steps per warp.
// Per warp step, ballots of the NB bits of each pair's expert (and, among the
// first pairs of their (token, rank), of its rank) give every lane x the
// lanes holding expert x (rank x) with one LOP per bit, so lane x owns the
// running counts of expert x and rank x; match.any gives a pair's rank among
// same-expert pairs and the (token, rank) duplicate test, and the token's
// rank bitmask is written straight to is_token_in_rank.  One CTA barrier
// turns the per-warp counts into warp bases (lanes split over experts and
// warps, xor-shuffle sums); warp q of each CTA then pushes its tile's counts
// into the shared memory of CTA q of the cluster (remote stores, no round trip),
// and after one cluster barrier every warp derives the tile prefixes, the
// totals and cu_seqlens from its own shared memory and writes its pairs'
// slots.  Tile 0's warp 0 writes the totals-derived outputs.  Per-pair
// results stay in registers.
constexpr int SMALL_MAX = 32;

__device__ __forceinline__ void st_dsmem_s32(uint32_t addr, int32_t v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int warp_incl_scan(int v, int width) {
    const int lane = threadIdx.x & 31;
    for (int off = 1; off < width; off <<= 1) {
        const int y = __shfl_up_sync(FULL_MASK, v, off);
        if (lane >= off) v += y;
    }
    return v;
}

// is_token_in_rank row of one token from its rank bitmask (bytes 0 / 1).
__device__ __forceinline__ void store_rank_row(uint8_t* row, uint32_t mask, int R) {
    if ((R & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 3u) == 0) {
        // bit i of a 4-bit m to byte i: m * (1 + 2^7 + 2^14 + 2^21) places
        // copies of m 7 bits apart (no carries), the mask keeps bit i of copy i
        for (int c = 0; c < R / 4; ++c)
            reinterpret_cast<uint32_t*>(row)[c] = (((mask >> (4 * c)) & 15u) * 0x204081u) & 0x01010101u;
    } else {
        for (int x = 0; x < R; ++x) row[x] = static_cast<uint8_t>((mask >> x) & 1u);
    }
}

// Where a warp's expert ids come from.  TopkSource: topk_idx, written by an
// earlier kernel.  RouteSource: routed here (the fused route + plan), one
// token per lane with route_token (the router's own arithmetic, so ids and
// weights are those of the routing kernel), the K winners written to
// topk_idx / topk_w and handed to the lanes of the (token, k) layout.
struct TopkSource {
    template <int IPT>
    __device__ __forceinline__ void fetch(const PlanArgs& a, int wt0, int lane, int tok_in_iter, int k, int act,
                                          int (&ids)[IPT]) const {
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int s = wt0 + i * a.tpw + tok_in_iter;
            ids[i] = (lane < act && s < a.N) ? __ldg(a.topk + s * a.K + k) : -1;
        }
    }
};

constexpr int FUSED_KMAX = 8;  // K <= 8 when routing inside the plan

// V logits per lane (float4 loads), V >= E, E % 4 == 0, K a power of two
// <= KM (2 or 8: the winners a lane holds), no group limit.  The warp's IPT steps cover IPT * 32 / K tokens,
// routed 32 at a time (chunk c: tokens wt0 + 32 c + lane); the steps of a
// chunk take their ids from it with K shuffles.
template <int V, int KM>
struct RouteSource {
    RouteArgs r;
    template <int IPT>
    __device__ __forceinline__ void fetch(const PlanArgs& a, int wt0, int lane, int tok_in_iter, int k, int act,
                                          int (&ids)[IPT]) const {
        const int K = a.K, tpw = a.tpw;
        float bias_r[V];
        lane_bias<1, V, true>(r, 0, bias_r);
        const int nt = IPT * tpw;  // tokens of this warp
#pragma unroll
        for (int i = 0; i < IPT; ++i) ids[i] = -1;
#pragma unroll
        for (int c = 0; c < IPT; ++c) {
            if (c * 32 >= nt) break;
            const int s = wt0 + c * 32 + lane;
            const bool valid = c * 32 + lane < nt && s < a.N;
            float raw[V];
            load_row<1, V, true>(r, valid ? s : a.N, 0, raw);
            int widx[KM];
            float wgt[KM];
            route_token<1, V, true, KM>(r, raw, bias_r, valid, lane, 0, nullptr, widx, wgt);
            if (valid) {
#pragma unroll
                for (int q = 0; q < KM; ++q)
                    if (q < K) {
                        r.topk_idx[static_cast<int64_t>(s) * K + q] = widx[q];
                        r.topk_w[static_cast<int64_t>(s) * K + q] = wgt[q];
                    }
            }
            // steps i whose tokens lie in this chunk: token i * tpw + tok_in_iter
            // of the warp sits in lane (i * tpw + tok_in_iter) mod 32
#pragma unroll
            for (int i = 0; i < IPT; ++i) {
                if ((i * tpw) / 32 != c) continue;  // uniform: tpw divides 32
                const int src = (i * tpw + tok_in_iter) & 31;
                int id = -1;
#pragma unroll
                for (int q = 0; q < KM; ++q) {
                    if (q >= K) break;
                    const int v = __shfl_sync(FULL_MASK, widx[q], src);
                    if (q == k) id = v;
                }
                const int st = wt0 + i * tpw + tok_in_iter;
                ids[i] = (lane < act && st < a.N) ? id : -1;
            }
        }
    }
};

template <int IPT, int NB, class Src>
__global__ void __launch_bounds__(PLAN_THREADS) plan_small_kernel(const PlanArgs a, const Src src) {
    constexpr int EP = 1 << NB;         // experts (and ranks) a lane group covers
    constexpr int CHUNKS = 32 / EP;     // lane groups per warp
    constexpr int CW = 2 * EP + 2;      // tile columns: experts, ranks, groups, duplicates
    constexpr int TPC = 16 / CHUNKS;    // tiles per lane group in the cross-tile sums
    __shared__ int32_t s_wc[PLAN_WARPS][EP + 1];  // per-warp pairs per expert (+1: no bank conflicts)
    __shared__ int32_t s_wr[PLAN_WARPS][EP + 1];  // per-warp tokens per rank
    __shared__ int32_t s_wg[PLAN_WARPS], s_wd[PLAN_WARPS];
    __shared__ int32_t s_all[16][CW];             // every tile's counts, pushed by its CTA

    // set-up that reads no memory of the previous kernels runs before the wait
    cluster_arrive_relaxed();  // this CTA has started: the others may push into it once all have
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E, K = a.K, R = a.R;
    const uint32_t crank = cluster_ctarank(), ncta = cluster_nctarank();
    const int tile = static_cast<int>(crank);
    const int tok0 = tile * a.tile_tokens;  // N * K < 2^30: token and pair indices fit in int
    const unsigned lt = (1u << lane) - 1u;
    const int act = a.tpw * K;
    const int tok_in_iter = lane / K, k = lane - tok_in_iter * K;
    const int tok_lane0 = tok_in_iter * K;
    const unsigned below_tok = (1u << tok_lane0) - 1u;
    const unsigned seg = (K >= 32 ? FULL_MASK : ((1u << K) - 1u)) << tok_lane0;  // the token's lanes
    const bool k_pow2 = (K & (K - 1)) == 0;
    unsigned xl[NB];  // bit b of this lane's index, as an all-ones / all-zeros word
#pragma unroll
    for (int b = 0; b < NB; ++b) xl[b] = 0u - ((static_cast<unsigned>(lane) >> b) & 1u);

    pdl_wait();
    pdl_trigger();
    int ids[IPT];
    src.template fetch<IPT>(a, tok0 + warp * IPT * a.tpw, lane, tok_in_iter, k, act, ids);

    // ---- first pass, all in registers
    int cnt_e = 0, cnt_r = 0, run_g = 0, run_d = 0;  // lane x: pairs of expert x / tokens on rank x so far
    uint2 item[IPT];
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
        const int s = tok0 + (warp * IPT + i) * a.tpw + tok_in_iter;
        bool active = lane < act && s < a.N;
        int e = 0;
        if (active) {
            e = ids[i];
            if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, s * K + k);
                active = false;
                e = 0;
            }
        }
        // bit b of every lane's expert and rank, one ballot each; lanes
        // holding a given value are the AND of matching bit words
        const unsigned amask = __ballot_sync(FULL_MASK, active);
        const int r = rank_of(a, e);
        unsigned me = amask, peers = amask, mr = amask, pr = amask;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const unsigned eb = __ballot_sync(FULL_MASK, (e >> b) & 1);
            const unsigned rb = __ballot_sync(FULL_MASK, (r >> b) & 1);
            me &= ~(eb ^ xl[b]);                   // lanes holding expert `lane`
            peers &= ~(eb ^ (0u - ((e >> b) & 1)));  // lanes holding this lane's expert
            mr &= ~(rb ^ xl[b]);                   // lanes on rank `lane`
            pr &= ~(rb ^ (0u - ((r >> b) & 1)));     // lanes on this lane's rank
        }
        const int wr = __popc(peers & lt) + __shfl_sync(FULL_MASK, cnt_e, e);
        cnt_e += __popc(me);

        const unsigned pd = pr & seg;  // this token's pairs on this lane's rank
        const bool prim = active && (pd & lt) == 0u;
        const bool dup = active && !prim;
        const bool opens = prim && __popc(pd) >= 2;
        const unsigned pmask = __ballot_sync(FULL_MASK, prim);
        cnt_r += __popc(mr & pmask);  // tokens on rank `lane`
        const unsigned gball = __ballot_sync(FULL_MASK, opens);
        const unsigned dball = amask & ~pmask;
        // duplicates of a token: group after group (groups in order of their
        // primary lane), k order inside a group; a warp scan of the group
        // sizes gives the duplicates of the groups opening before a lane
        int groups_before = 0;  // with K <= 2 a token has at most one group
        if (K > 2) {
            const int my_p = __ffs(pd) - 1;
            const int gsz = opens ? __popc(pd) - 1 : 0;
            const int excl = warp_incl_scan(gsz, 32) - gsz;
            const int tok_base = __shfl_sync(FULL_MASK, excl, tok_lane0 & 31);
            groups_before = __shfl_sync(FULL_MASK, excl, my_p & 31) - tok_base;
        }
        const int before = groups_before + (dup ? __popc(pd & lt) - 1 : 0);
        const int dup_pos = run_d + __popc(dball & below_tok) + before;

        // the token's rank bitmask: OR over its K lanes
        uint32_t rbits = prim ? 1u << r : 0u;
        if (k_pow2) {
            for (int off = 1; off < K; off <<= 1) rbits |= __shfl_xor_sync(FULL_MASK, rbits, off);
        } else {
            uint32_t acc = 0;
            for (int q = 0; q < K; ++q) acc |= __shfl_sync(FULL_MASK, rbits, (tok_lane0 + q) & 31);
            rbits = acc;
        }
        if (active && k == 0) store_rank_row(a.out.is_token_in_rank + static_cast<int64_t>(s) * R, rbits, R);

        item[i] = active ? pack_item(e, wr, dup, opens, __popc(pd) - 1, opens ? run_g + __popc(gball & lt) : dup_pos,
                                     dup_pos)
                         : make_uint2(ITEM_NONE, 0u);
        run_g += __popc(gball);
        run_d += __popc(dball);
    }
    if (lane < EP) {
        s_wc[warp][lane] = cnt_e;
        s_wr[warp][lane] = cnt_r;
    }
    if (lane == 0) {
        s_wg[warp] = run_g;
        s_wd[warp] = run_d;
    }
    __syncthreads();
    cluster_wait();  // every CTA of the cluster has started

    // ---- warp bases: lane l sums expert (l mod EP) over warps
    // [(l / EP) * EP, +EP), then xor-shuffles add the lane groups
    const int x = lane & (EP - 1), chunk = lane / EP;
    int base_e = 0, tile_e = 0;
    {
        int v[EP];
#pragma unroll
        for (int j = 0; j < EP; ++j) v[j] = s_wc[chunk * EP + j][x];
#pragma unroll
        for (int j = 0; j < EP; ++j) {
            base_e += chunk * EP + j < warp ? v[j] : 0;
            tile_e += v[j];
        }
#pragma unroll
        for (int off = EP; off < 32; off <<= 1) {
            base_e += __shfl_xor_sync(FULL_MASK, base_e, off);
            tile_e += __shfl_xor_sync(FULL_MASK, tile_e, off);
        }
    }
    const int vg = s_wg[lane], vd = s_wd[lane];  // PLAN_WARPS == 32
    const int g_wbase = __reduce_add_sync(FULL_MASK, lane < warp ? vg : 0);
    const int d_wbase = __reduce_add_sync(FULL_MASK, lane < warp ? vd : 0);

    // ---- the tile's counts; warp q pushes them into CTA q's s_all[tile]
    if (static_cast<uint32_t>(warp) < ncta) {
        int tile_r = 0;
        {
            int v[EP];
#pragma unroll
            for (int j = 0; j < EP; ++j) v[j] = s_wr[chunk * EP + j][x];
#pragma unroll
            for (int j = 0; j < EP; ++j) tile_r += v[j];
#pragma unroll
            for (int off = EP; off < 32; off <<= 1) tile_r += __shfl_xor_sync(FULL_MASK, tile_r, off);
        }
        const int g_tile = __reduce_add_sync(FULL_MASK, vg), d_tile = __reduce_add_sync(FULL_MASK, vd);
#pragma unroll
        for (int c0 = 0; c0 < CW; c0 += 32) {
            const int c = c0 + lane;
            const int ve = __shfl_sync(FULL_MASK, tile_e, c & (EP - 1));
            const int vr = __shfl_sync(FULL_MASK, tile_r, (c - EP) & (EP - 1));
            const int val = c < EP ? ve : c < 2 * EP ? vr : c == 2 * EP ? g_tile : d_tile;
            if (c < CW) st_dsmem_s32(dsmem_addr(&s_all[tile][c], static_cast<uint32_t>(warp)), val);
        }
    }
    cluster_arrive();  // release: this CTA's pushes
    cluster_wait();    // acquire: every tile's counts are in s_all

    // ---- lower tiles and totals, every warp from its own shared memory
    int pre_e = 0, tot_e = 0;
    {
#pragma unroll
        for (int j = 0; j < TPC; ++j) {
            const int q = chunk * TPC + j;
            const int v = q < static_cast<int>(ncta) ? s_all[q][x] : 0;
            pre_e += q < tile ? v : 0;
            tot_e += v;
        }
#pragma unroll
        for (int off = EP; off < 32; off <<= 1) {
            pre_e += __shfl_xor_sync(FULL_MASK, pre_e, off);
            tot_e += __shfl_xor_sync(FULL_MASK, tot_e, off);
        }
    }
    int gq = 0, dq = 0;
    if (static_cast<uint32_t>(lane) < ncta) {
        gq = s_all[lane][2 * EP];
        dq = s_all[lane][2 * EP + 1];
    }
    const int g_pre = __reduce_add_sync(FULL_MASK, lane < tile ? gq : 0);
    const int d_pre = __reduce_add_sync(FULL_MASK, lane < tile ? dq : 0);

    const unsigned al = static_cast<unsigned>(a.alignment);
    int padded = 0;
    if (lane < E && tot_e > 0) {
        const unsigned t = static_cast<unsigned>(tot_e) + al - 1u;
        padded = static_cast<int>((al & (al - 1u)) == 0u ? (t & ~(al - 1u)) : t / al * al);
    }
    const int cu_incl = warp_incl_scan(padded, EP);
    const int cu_e = cu_incl - padded;
    const int P = __shfl_sync(FULL_MASK, cu_incl, EP - 1);
    const int slot_base = cu_e + pre_e + base_e;  // first slot of expert `lane` in this warp run

    // ---- second pass: slots, dst, src_of_slot, dedup structures
    const int64_t gbase = static_cast<int64_t>(g_pre) + g_wbase, dbase = static_cast<int64_t>(d_pre) + d_wbase;
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
        const uint2 it = item[i];
        const uint32_t e = it.x & 0x7ffu;
        const int sb = __shfl_sync(FULL_MASK, slot_base, static_cast<int>(e & 31u));
        if (e == ITEM_NONE) continue;
        const int s = tok0 + (warp * IPT + i) * a.tpw + tok_in_iter;
        const int f = s * K + k;
        const int32_t slot = sb + static_cast<int32_t>((it.x >> 11) & 0x3ffu);
        if (slot < 0 || static_cast<int64_t>(slot) >= a.p_cap) {
            record_error(a.out.status, MOE_ERR_DEVICE_INDEX, slot);
            continue;
        }
        const bool dup = (it.x >> 21) & 1u;
        const bool opens = (it.x >> 22) & 1u;
        const int32_t ia = static_cast<int32_t>(it.y & 0xffffu), ib = static_cast<int32_t>(it.y >> 16);
        a.out.dst[f] = dup ? -slot - 1 : slot;
        a.out.src_of_slot[slot] = f;
        if (opens) {
            const int64_t g = gbase + ia;
            if (g >= static_cast<int64_t>(a.N) * (K / 2)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(g));
                continue;
            }
            int32_t* row = a.out.dup_groups + 3 * g;
            row[0] = slot;
            row[1] = static_cast<int32_t>(dbase + ib);
            row[2] = static_cast<int32_t>(it.x >> 23);
        } else if (dup) {
            const int64_t pos = dbase + ia;
            if (pos >= static_cast<int64_t>(a.N) * (K - 1)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(pos));
                continue;
            }
            a.out.dup_loffs[pos] = slot;
        }
    }

    // ---- totals-derived outputs (MoonEP cu_seqlens / zero_fill_ranges;
    // DeepEP notify_dispatch rank prefix)
    if (tile == 0 && warp == 0) {
        int tot_r = 0;
#pragma unroll
        for (int j = 0; j < TPC; ++j) {
            const int q = chunk * TPC + j;
            tot_r += q < static_cast<int>(ncta) ? s_all[q][EP + x] : 0;
        }
#pragma unroll
        for (int off = EP; off < 32; off <<= 1) tot_r += __shfl_xor_sync(FULL_MASK, tot_r, off);
        if (lane >= R) tot_r = 0;
        const int32_t g_tot = __reduce_add_sync(FULL_MASK, gq), d_tot = __reduce_add_sync(FULL_MASK, dq);
        const int epn = a.epn;
        const int rso = __shfl_sync(FULL_MASK, cu_e, (lane * epn) & 31);
        int ppr = 0;
        for (int j = 0; j < epn; ++j) ppr += __shfl_sync(FULL_MASK, tot_e, (lane * epn + j) & 31);
        const int tpr_incl = warp_incl_scan(tot_r, 32);
        const int tpr_total = __shfl_sync(FULL_MASK, tpr_incl, 31);
        if (lane < E) {
            a.out.tokens_per_expert[lane] = tot_e;
            a.out.cu_seqlens[lane] = cu_e;
            const int pad = padded - tot_e;
            a.out.zero_fill_ranges[2 * lane] = pad > 0 ? cu_e + tot_e : 0;
            a.out.zero_fill_ranges[2 * lane + 1] = pad > 0 ? pad : 0;
        }
        if (lane < R) {
            a.out.rank_slot_offsets[lane] = rso;
            a.out.pairs_per_rank[lane] = ppr;
            a.out.tokens_per_rank[lane] = tot_r;
            a.out.rank_prefix[lane] = tpr_incl - tot_r;
        }
        if (lane == 0) {
            a.out.cu_seqlens[E] = P;
            a.out.rank_slot_offsets[R] = P;
            a.out.rank_prefix[R] = tpr_total;
            a.out.dup_counts[0] = g_tot;
            a.out.dup_counts[1] = d_tot;
        }
    }

    // ---- -1 into the padding rows (warp w: expert w, on tiles w mod T)
    // and into this tile's share of the unused rows [P, P_cap)
    if (warp < E && static_cast<uint32_t>(warp) % ncta == crank) {
        const int start = __shfl_sync(FULL_MASK, cu_e + tot_e, warp);
        const int end = __shfl_sync(FULL_MASK, cu_incl, warp);
        for (int j = start + lane; j < end; j += 32)
            if (j >= 0 && static_cast<int64_t>(j) < a.p_cap) a.out.src_of_slot[j] = -1;
    }
    {
        const uint32_t cap = static_cast<uint32_t>(a.p_cap);  // < 2^31
        const uint32_t rest = cap - static_cast<uint32_t>(P);
        const uint32_t share = (rest + ncta - 1u) / ncta;
        const uint32_t b = static_cast<uint32_t>(P) + share * crank, e = min(cap, b + share);
        for (uint32_t j = b + tid; j < e; j += PLAN_THREADS) a.out.src_of_slot[j] = -1;
    }
}

// ---------------------------------------------------------------- medium-E path
// 32 < E <= 32 * EW (EW = 4 or 8) and R <= 32: the small-E scheme, except
// that each warp keeps its running pairs per expert in a shared-memory row:
// per warp step, match.any gives a pair the lanes holding its expert (at
// this E cheaper than the bit ballots: the step is bound by the integer
// pipe), it reads its expert's running count (lanes of a group read one
// word) and the group's first lane writes the new count back.
// After the first pass one CTA-wide column scan turns the [32 warps][E]
// counts into warp bases: thread (e, q) scans expert e over warps
// [8q, 8q + 8), a second barrier adds the quarter offsets and yields the
// tile count, which the thread pushes into four CTAs of the cluster.  After
// the cluster barrier threads e < E derive the expert's tile prefix and
// total, warp 0 scans the padded totals into cu_seqlens, and the second
// pass writes the slots.  Per-pair results stay in registers.
template <int IPT, int EW>
__global__ void __launch_bounds__(PLAN_THREADS) plan_medium_kernel(const PlanArgs a) {
    constexpr int NBR = 5;  // rank bits (R <= 32)
    extern __shared__ __align__(16) int32_t s_dyn[];
    const int E = a.E, K = a.K, R = a.R, C = a.C;
    int32_t* s_wc = s_dyn;                       // [32][E]   per-warp pairs per expert, then warp bases
    int32_t* s_qt = s_wc + PLAN_WARPS * E;       // [4][256]  per-quarter totals
    int32_t* s_all = s_qt + 4 * 256;             // [16][C]   every tile's counts, pushed by its CTA
    int32_t* s_base = s_all + 16 * C;            // [E]       cu[e] + pairs of e in lower tiles
    int32_t* s_pad = s_base + E;                 // [E]       padded totals, then cu_seqlens
    int32_t* s_tot = s_pad + E;                  // [E]       totals
    int32_t* s_src = s_tot + E;                  // [32 * IPT * 32] the tile's pairs in slot order: f
    int32_t* s_gsl = s_src + PLAN_WARPS * 32 * IPT;  // [32 * IPT * 32] ... and their slots
    int32_t* s_tloc = s_qt;                      // [E + 1]   tile-local first pair per expert (after the exchange)
    __shared__ int32_t s_wr[PLAN_WARPS][SMALL_MAX + 1];
    __shared__ int32_t s_wg[PLAN_WARPS], s_wd[PLAN_WARPS];
    __shared__ int32_t s_gd[4];  // groups, duplicates of lower tiles; their totals

    cluster_arrive_relaxed();  // this CTA has started: the others may push into it once all have
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t crank = cluster_ctarank(), ncta = cluster_nctarank();
    const int tile = static_cast<int>(crank);
    const int tok0 = tile * a.tile_tokens;  // N * K < 2^30: token and pair indices fit in int
    const unsigned lt = (1u << lane) - 1u;
    const int act = a.tpw * K;
    const int tok_in_iter = lane / K, k = lane - tok_in_iter * K;
    const int tok_lane0 = tok_in_iter * K;
    const unsigned below_tok = (1u << tok_lane0) - 1u;
    const unsigned seg = (K >= 32 ? FULL_MASK : ((1u << K) - 1u)) << tok_lane0;
    const bool k_pow2 = (K & (K - 1)) == 0;
    unsigned xl[5];
#pragma unroll
    for (int b = 0; b < 5; ++b) xl[b] = 0u - ((static_cast<unsigned>(lane) >> b) & 1u);
    const int rbits = R > 1 ? 32 - __clz(R - 1) : 0;  // rank bits in use
    int32_t* wrow = s_wc + warp * E;  // this warp's running pairs per expert
    for (int e = lane; e < E; e += 32) wrow[e] = 0;
    __syncwarp();

    pdl_wait();
    pdl_trigger();
    int ids[IPT];
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
        const int s = tok0 + (warp * IPT + i) * a.tpw + tok_in_iter;
        ids[i] = (lane < act && s < a.N) ? __ldg(a.topk + s * K + k) : -1;
    }

    // ---- first pass: per-pair results in registers, running counts per
    // expert in the warp's shared row (the group's first lane writes back)
    int cnt_r = 0, run_g = 0, run_d = 0;
    uint2 item[IPT];
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
        const int s = tok0 + (warp * IPT + i) * a.tpw + tok_in_iter;
        bool active = lane < act && s < a.N;
        int e = 0;
        if (active) {
            e = ids[i];
            if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, s * K + k);
                active = false;
                e = 0;
            }
        }
        const unsigned amask = __ballot_sync(FULL_MASK, active);
        const int r = rank_of(a, e);
        // with E in the hundreds one match beats NBE ballots and their LOPs
        const unsigned peers = __match_any_sync(FULL_MASK, active ? e : -1);
        unsigned pr = amask, mr = amask;
#pragma unroll
        for (int b = 0; b < NBR; ++b) {
            const unsigned rb = b < rbits ? __ballot_sync(FULL_MASK, (r >> b) & 1) : 0u;
            mr &= ~(rb ^ xl[b]);
            pr &= ~(rb ^ (0u - ((r >> b) & 1)));
        }
        const int base = active ? wrow[e] : 0;
        __syncwarp();
        if (active && (peers & lt) == 0u) wrow[e] = base + __popc(peers);
        __syncwarp();
        const int wr = base + __popc(peers & lt);

        const unsigned pd = pr & seg;  // this token's pairs on this lane's rank
        const bool prim = active && (pd & lt) == 0u;
        const bool dup = active && !prim;
        const bool opens = prim && __popc(pd) >= 2;
        const unsigned pmask = __ballot_sync(FULL_MASK, prim);
        cnt_r += __popc(mr & pmask);
        const unsigned gball = __ballot_sync(FULL_MASK, opens);
        const unsigned dball = amask & ~pmask;
        int groups_before = 0;
        if (K > 2) {
            const int my_p = __ffs(pd) - 1;
            const int gsz = opens ? __popc(pd) - 1 : 0;
            const int excl = warp_incl_scan(gsz, 32) - gsz;
            const int tok_base = __shfl_sync(FULL_MASK, excl, tok_lane0 & 31);
            groups_before = __shfl_sync(FULL_MASK, excl, my_p & 31) - tok_base;
        }
        const int before = groups_before + (dup ? __popc(pd & lt) - 1 : 0);
        const int dup_pos = run_d + __popc(dball & below_tok) + before;

        uint32_t rbits = prim ? 1u << r : 0u;
        if (k_pow2) {
            for (int off = 1; off < K; off <<= 1) rbits |= __shfl_xor_sync(FULL_MASK, rbits, off);
        } else {
            uint32_t acc = 0;
            for (int q = 0; q < K; ++q) acc |= __shfl_sync(FULL_MASK, rbits, (tok_lane0 + q) & 31);
            rbits = acc;
        }
        if (active && k == 0) store_rank_row(a.out.is_token_in_rank + static_cast<int64_t>(s) * R, rbits, R);

        item[i] = active ? pack_item(e, wr, dup, opens, __popc(pd) - 1, opens ? run_g + __popc(gball & lt) : dup_pos,
                                     dup_pos)
                         : make_uint2(ITEM_NONE, 0u);
        run_g += __popc(gball);
        run_d += __popc(dball);
    }
    s_wr[warp][lane] = cnt_r;
    if (lane == 0) {
        s_wg[warp] = run_g;
        s_wd[warp] = run_d;
    }
    // -1 over this CTA's share of every row of src_of_slot; the pairs' rows
    // are written after the cluster barrier below (release / acquire), so
    // they land after these, and the padding and unused rows keep -1
    {
        const uint32_t cap = static_cast<uint32_t>(a.p_cap);  // < 2^31
        const uint32_t share = (cap + ncta - 1u) / ncta;
        const uint32_t b = share * crank, e = min(cap, b + share);
        for (uint32_t j = b + tid; j < e; j += PLAN_THREADS) a.out.src_of_slot[j] = -1;
    }
    __syncthreads();
    cluster_wait();  // every CTA of the cluster has started

    // ---- column scan over warps: thread (e, q) takes warps [8q, 8q + 8)
    const int ce = tid & 255, cq = tid >> 8;
    int v[8];
    int qsum = 0;
    if (ce < E) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = s_wc[(8 * cq + i) * E + ce];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = v[i];
            v[i] = qsum;  // exclusive within the quarter
            qsum += c;
        }
        s_qt[cq * 256 + ce] = qsum;
    }
    // groups and duplicates: warp 1 scans the warp runs (bases kept in s_wg / s_wd)
    if (warp == 1) {
        const int g = s_wg[lane], d = s_wd[lane];
        const int gi = warp_incl_scan(g, 32), di = warp_incl_scan(d, 32);
        s_wg[lane] = gi - g;
        s_wd[lane] = di - d;
        if (lane == 31) {
            s_gd[2] = gi;  // this tile's groups and duplicates
            s_gd[3] = di;
        }
    }
    int tile_r = 0;
    if (warp == 2) {
#pragma unroll 8
        for (int w = 0; w < PLAN_WARPS; ++w) tile_r += s_wr[w][lane];
    }
    __syncthreads();

    // ---- quarter offsets -> warp bases; tile counts pushed to the cluster
    if (ce < E) {
        int qoff = 0, tile_e = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int t = s_qt[q * 256 + ce];
            qoff += q < cq ? t : 0;
            tile_e += t;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) s_wc[(8 * cq + i) * E + ce] = v[i] + qoff;
        for (uint32_t q = static_cast<uint32_t>(cq); q < ncta; q += 4)
            st_dsmem_s32(dsmem_addr(s_all + tile * C + ce, q), tile_e);
    }
    if (warp == 2) {  // ranks: lane r pushes to every CTA
        if (lane < R)
            for (uint32_t q = 0; q < ncta; ++q) st_dsmem_s32(dsmem_addr(s_all + tile * C + E + lane, q), tile_r);
    }
    if (warp == 3 && static_cast<uint32_t>(lane) < ncta) {  // groups, duplicates: lane q pushes to CTA q
        st_dsmem_s32(dsmem_addr(s_all + tile * C + E + R, lane), s_gd[2]);
        st_dsmem_s32(dsmem_addr(s_all + tile * C + E + R + 1, lane), s_gd[3]);
    }
    cluster_arrive();  // release: this CTA's pushes
    cluster_wait();    // acquire: every tile's counts are in s_all

    // ---- lower tiles and totals per expert; groups / duplicates of lower tiles
    const int al = a.alignment;
    for (int e = tid; e < E; e += PLAN_THREADS) {
        int pre = 0, tot = 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const int t = q < static_cast<int>(ncta) ? s_all[q * C + e] : 0;
            pre += q < tile ? t : 0;
            tot += t;
        }
        s_base[e] = pre;
        s_tot[e] = tot;
        const unsigned u = static_cast<unsigned>(tot) + static_cast<unsigned>(al) - 1u;
        const unsigned alu = static_cast<unsigned>(al);
        s_pad[e] = tot > 0 ? static_cast<int>((alu & (alu - 1u)) == 0u ? (u & ~(alu - 1u)) : u / alu * alu) : 0;
    }
    if (warp == PLAN_WARPS - 1) {
        const int gq = static_cast<uint32_t>(lane) < ncta ? s_all[lane * C + E + R] : 0;
        const int dq = static_cast<uint32_t>(lane) < ncta ? s_all[lane * C + E + R + 1] : 0;
        const int gp = __reduce_add_sync(FULL_MASK, lane < tile ? gq : 0);
        const int dp = __reduce_add_sync(FULL_MASK, lane < tile ? dq : 0);
        const int gt = __reduce_add_sync(FULL_MASK, gq), dt = __reduce_add_sync(FULL_MASK, dq);
        if (lane == 0) {
            s_gd[0] = gp;
            s_gd[1] = dp;
            if (tile == 0) {
                a.out.dup_counts[0] = gt;
                a.out.dup_counts[1] = dt;
            }
        }
    }
    __syncthreads();

    // ---- warp 0: cu_seqlens (lane l scans experts [l * EW, l * EW + EW)),
    // tile 0 also the totals-derived outputs
    if (warp == 0) {
        int pv[EW], tv[EW], run = 0, trun = 0;
#pragma unroll
        for (int j = 0; j < EW; ++j) {
            const int e = lane * EW + j;
            pv[j] = e < E ? s_pad[e] : 0;
            tv[j] = e < E ? s_all[tile * C + e] : 0;
            run += pv[j];
            trun += tv[j];
        }
        const int incl = warp_incl_scan(run, 32);
        int c = incl - run;
        const int P = __shfl_sync(FULL_MASK, incl, 31);
        const int tincl = warp_incl_scan(trun, 32);
        int tl = tincl - trun;
#pragma unroll
        for (int j = 0; j < EW; ++j) {
            const int e = lane * EW + j;
            if (e < E) s_tloc[e] = tl;
            tl += tv[j];
        }
        if (lane == 31) s_tloc[E] = tincl;
#pragma unroll
        for (int j = 0; j < EW; ++j) {
            const int e = lane * EW + j;
            if (e < E) {
                if (tile == 0) {
                    const int tot = s_tot[e];
                    a.out.tokens_per_expert[e] = tot;
                    a.out.cu_seqlens[e] = c;
                    const int pad = pv[j] - tot;
                    a.out.zero_fill_ranges[2 * e] = pad > 0 ? c + tot : 0;
                    a.out.zero_fill_ranges[2 * e + 1] = pad > 0 ? pad : 0;
                }
                s_base[e] += c;
                s_pad[e] = c;  // s_pad now holds cu_seqlens
            }
            c += pv[j];
        }
        if (tile == 0 && lane == 0) {
            a.out.cu_seqlens[E] = P;
            a.out.rank_slot_offsets[R] = P;
        }
    }
    __syncthreads();

    if (tile == 0 && warp == 1) {  // rank arrays (DeepEP notify_dispatch rank prefix)
        int tot_r = 0;
        if (lane < R)
            for (int q = 0; q < static_cast<int>(ncta); ++q) tot_r += s_all[q * C + E + lane];
        const int incl = warp_incl_scan(tot_r, 32);
        const int total = __shfl_sync(FULL_MASK, incl, 31);
        if (lane < R) {
            int ppr = 0;
            for (int e = lane * a.epn; e < (lane + 1) * a.epn; ++e) ppr += s_tot[e];
            a.out.rank_slot_offsets[lane] = s_pad[lane * a.epn];
            a.out.pairs_per_rank[lane] = ppr;
            a.out.tokens_per_rank[lane] = tot_r;
            a.out.rank_prefix[lane] = incl - tot_r;
        }
        if (lane == 0) a.out.rank_prefix[R] = total;
    }

    // ---- second pass: slots, dst, src_of_slot, dedup structures
    const int64_t gbase = static_cast<int64_t>(s_gd[0]) + s_wg[warp];
    const int64_t dbase = static_cast<int64_t>(s_gd[1]) + s_wd[warp];
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
        const uint2 it = item[i];
        const uint32_t e = it.x & 0x7ffu;
        if (e == ITEM_NONE) continue;
        const int s = tok0 + (warp * IPT + i) * a.tpw + tok_in_iter;
        const int f = s * K + k;
        const int32_t in_tile = s_wc[warp * E + e] + static_cast<int32_t>((it.x >> 11) & 0x3ffu);
        const int32_t slot = s_base[e] + in_tile;
        if (slot < 0 || static_cast<int64_t>(slot) >= a.p_cap) {
            record_error(a.out.status, MOE_ERR_DEVICE_INDEX, slot);
            continue;
        }
        s_src[s_tloc[e] + in_tile] = f;
        s_gsl[s_tloc[e] + in_tile] = slot;
        const bool dup = (it.x >> 21) & 1u;
        const bool opens = (it.x >> 22) & 1u;
        const int32_t ia = static_cast<int32_t>(it.y & 0xffffu), ib = static_cast<int32_t>(it.y >> 16);
        a.out.dst[f] = dup ? -slot - 1 : slot;
        if (opens) {
            const int64_t g = gbase + ia;
            if (g >= static_cast<int64_t>(a.N) * (K / 2)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(g));
                continue;
            }
            int32_t* row = a.out.dup_groups + 3 * g;
            row[0] = slot;
            row[1] = static_cast<int32_t>(dbase + ib);
            row[2] = static_cast<int32_t>(it.x >> 23);
        } else if (dup) {
            const int64_t pos = dbase + ia;
            if (pos >= static_cast<int64_t>(a.N) * (K - 1)) {
                record_error(a.out.status, MOE_ERR_DEVICE_INDEX, static_cast<int>(pos));
                continue;
            }
            a.out.dup_loffs[pos] = slot;
        }
    }

    // ---- src_of_slot: each expert's pairs of this tile are one run of
    // slots, staged in slot order, so neighbouring threads store
    // neighbouring slots
    __syncthreads();
    for (int i = tid; i < s_tloc[E]; i += PLAN_THREADS) a.out.src_of_slot[s_gsl[i]] = s_src[i];
}

// ---------------------------------------------------------------- grid path
// The whole plan in one launch of T <= 152 CTAs of WARPS warps, all resident
// at once (the host checks the occupancy), one tile each.  Each CTA runs its
// tile's first pass and publishes the column counts column-major
// (counts[c][tile]) followed by one epoch-tagged flag word; then it waits
// (bounded in time) until every tile's flag carries the running call's tag
// and reduces every tile's counts itself: the sum over lower tiles is its
// exclusive prefix, the sum over all the totals.  Every CTA scans the totals
// into cu_seqlens, tile 0 writes the totals-derived outputs, and the tile's
// second pass writes the slots.  The last CTA to finish closes the epoch.
// Compared with the cluster path the work is spread over all SMs; compared
// with the look-back path there is no chain of waits and one launch.
template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32) plan_grid_kernel(const PlanArgs a) {
    constexpr int THREADS = WARPS * 32;
    extern __shared__ __align__(16) int32_t s_dyn[];
    const int E = a.E, R = a.R, C = a.C, T = a.T;
    uint2* s_items = reinterpret_cast<uint2*>(s_dyn);  // [WARPS][ipt][32]
    int32_t* s_wc = s_dyn + 2 * WARPS * 32 * a.ipt;     // [WARPS][E]
    int32_t* s_cnt = s_wc + WARPS * E;                  // [C]  this tile's column counts
    int32_t* s_tot = s_cnt + C;                         // [C]  totals over all tiles
    int32_t* s_excl = s_tot + C;                        // [C]  sums over lower tiles
    int32_t* s_pad = s_excl + C;                        // [E + R + 2]
    int32_t* s_cu = s_pad + E + R + 2;                  // [E + R + 2]
    uint8_t* s_itr = align16_after(s_dyn, s_cu + E + R + 2);  // [tile_tokens][R]
    __shared__ int32_t s_wg[WARPS], s_wd[WARPS], s_warp[WARPS + 1];
    __shared__ uint32_t s_epoch;
    __shared__ int s_bad;

    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.x;
    if (tid == 0) {
        // the ticket only validates the header: a workspace that was never
        // zeroed hands out an id outside [0, T) to some CTA
        const uint32_t ticket = atomicAdd(&a.hdr->ticket, 1u);
        s_epoch = (*reinterpret_cast<volatile uint32_t*>(&a.hdr->epoch) + 1u) & 0x7fffffffu;
        s_bad = ticket >= static_cast<uint32_t>(T) ? 1 : 0;
        if (s_bad) record_error(a.out.status, MOE_ERR_WORKSPACE, static_cast<int>(ticket));
    }
    const int itr_bytes = a.tile_tokens * R;
    for (int i = tid; i < WARPS * E; i += THREADS) s_wc[i] = 0;
    for (int i = tid; i < (itr_bytes + 3) / 4; i += THREADS) reinterpret_cast<int32_t*>(s_itr)[i] = 0;
    for (int c = E + tid; c < C; c += THREADS) s_cnt[c] = 0;
    __syncthreads();
    const uint32_t epoch = s_epoch;

    tile_phase1(a, tile, s_wc, s_itr, s_wg, s_wd, s_cnt + E, s_items);
    __syncthreads();
    for (int e = tid; e < E; e += THREADS) {
        int32_t v[WARPS];
#pragma unroll
        for (int w = 0; w < WARPS; ++w) v[w] = s_wc[w * E + e];
        int32_t c = 0;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) c += v[w];
        s_cnt[e] = c;
    }
    if (warp == 0) {
        const int32_t g = __reduce_add_sync(FULL_MASK, lane < WARPS ? s_wg[lane] : 0);
        const int32_t d = __reduce_add_sync(FULL_MASK, lane < WARPS ? s_wd[lane] : 0);
        if (lane == 0) {
            s_cnt[E + R] = g;
            s_cnt[E + R + 1] = d;
        }
    }
    __syncthreads();

    // ---- publish: counts, then the flag (every writer fences before the
    // barrier, so the flag store is ordered after all of them)
    int32_t* counts = a.tile_prefix;  // [C][T], T padded to a multiple of 4
    const int TP = (T + 3) & ~3;
    for (int c = tid; c < C; c += THREADS) st_relaxed_s32(counts + static_cast<size_t>(c) * TP + tile, s_cnt[c]);
    __syncthreads();
    // one fence after the barrier orders every thread's count stores (the
    // barrier makes them observed by thread 0; fences are cumulative)
    if (tid == 0 && tile != a.skip_tile) {
        __threadfence();
        st_relaxed_u64(a.flags + tile, pack_flag(epoch, s_bad ? ST_ERR : ST_PRE, 0u));
    }

    // ---- wait for every tile's flag (a thread per tile; T <= THREADS)
    if (tid < T) {
        uint64_t t0 = 0;
        while (true) {
            const uint64_t w = ld_relaxed_u64(a.flags + tid);
            if (static_cast<uint32_t>(w >> 32) == flag_tag(epoch)) {
                if (((static_cast<uint32_t>(w) >> 30) & 3u) == ST_ERR) s_bad = 1;
                break;
            }
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > static_cast<uint64_t>(a.timeout_ns)) {
                record_error(a.out.status, MOE_ERR_DEVICE_TIMEOUT, tile);
                s_bad = 1;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();  // acquire: the counts behind the flag are read below
    }
    __syncthreads();

    if (!s_bad) {  // uniform across the CTA
        // ---- every tile's counts: a warp per column, lanes over tiles;
        // the per-rank columns are needed by tile 0 only
        for (int c = warp; c < C; c += WARPS) {
            if (tile != 0 && c >= E && c < E + R) continue;
            const int32_t* col = counts + static_cast<size_t>(c) * TP;
            int32_t tot = 0, ex = 0;
            // 16-byte loads at L2 (past L1, written by other SMs): one
            // round trip per column for T <= 128
            for (int j = 4 * lane; j < T; j += 128) {
                const int4 v = __ldcg(reinterpret_cast<const int4*>(col + j));
                const int32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (j + u < T) {
                        tot += x[u];
                        ex += j + u < tile ? x[u] : 0;
                    }
                }
            }
            tot = __reduce_add_sync(FULL_MASK, tot);
            ex = __reduce_add_sync(FULL_MASK, ex);
            if (lane == 0) {
                s_tot[c] = tot;
                s_excl[c] = ex;
            }
        }
        __syncthreads();
        plan_totals<WARPS>(a, s_tot, s_pad, s_cu, s_warp, tile == 0);
        for (int e = tid; e < E; e += THREADS) s_excl[e] += s_cu[e];  // first slot of e in this tile
        __syncthreads();
        tile_phase3<WARPS>(a, tile, s_excl, s_excl[E + R], s_excl[E + R + 1], s_wc, s_wg, s_wd, s_itr, s_items);
        fill_unused<WARPS>(a, tile, T, s_cu, s_tot);
    }

    // ---- completion: the last CTA to finish closes the epoch
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&a.hdr->done, 1u);
        if (prev == gridDim.x - 1) {
            a.hdr->ticket = 0u;
            a.hdr->done = 0u;
            a.hdr->epoch = epoch;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------- empty batch
// N = 0 (a batch with no tokens): every count, offset and prefix is zero,
// no expert has padding, and every row of the capacity E * (alignment - 1)
// is unused (-1).  The arrays sized by N have no elements.
__global__ void __launch_bounds__(256) plan_empty_kernel(const MoePlanOut out, int E, int R, int64_t p_cap) {
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i <= E; i += blockDim.x) {
            out.cu_seqlens[i] = 0;
            if (i < E) {
                out.tokens_per_expert[i] = 0;
                out.zero_fill_ranges[2 * i] = 0;
                out.zero_fill_ranges[2 * i + 1] = 0;
            }
        }
        for (int i = threadIdx.x; i <= R; i += blockDim.x) {
            out.rank_prefix[i] = 0;
            out.rank_slot_offsets[i] = 0;
            if (i < R) {
                out.pairs_per_rank[i] = 0;
                out.tokens_per_rank[i] = 0;
            }
        }
        if (threadIdx.x < 2) out.dup_counts[threadIdx.x] = 0;
    }
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < p_cap; j += stride)
        out.src_of_slot[j] = -1;
}

}  // namespace moe

// ---------------------------------------------------------------- host
namespace {

using moe::PlanArgs;

struct Geom {
    int tpw, ipt, tile_tokens, T, C;
};

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return v ? std::atoi(v) : dflt;
}

Geom plan_geometry(int N, int E, int K, int R) {
    Geom g;
    g.tpw = 32 / K;
    const int64_t pairs = static_cast<int64_t>(N) * K;
    const int64_t per_iter = static_cast<int64_t>(moe::PLAN_WARPS) * g.tpw * K;
    // about one tile per SM of a GB300 (152 SMs); fixed so that the workspace
    // size is a function of the sizes alone
    constexpr int64_t kTargetTiles = 152;
    int64_t ipt = (pairs + per_iter * kTargetTiles - 1) / (per_iter * kTargetTiles);
    if (ipt < 1) ipt = 1;
    if (ipt > moe::PLAN_IPT_MAX) ipt = moe::PLAN_IPT_MAX;
    // shared memory of the scatter kernel: per-pair items, per-warp expert
    // counts, the tile's is_token_in_rank rows; shrink steps, then tokens per
    // step, until it fits and the rows stay within 64 KB
    auto smem2 = [&](int64_t st, int64_t tpw) {
        return 4 * (2 * moe::PLAN_WARPS * 32 * st + static_cast<int64_t>(moe::PLAN_WARPS + 1) * E + 4) +
               (moe::PLAN_WARPS * st * tpw * R + 15) / 16 * 16;
    };
    constexpr int64_t kSmemBudget = 220 * 1024;
    while (ipt > 1 && (static_cast<int64_t>(moe::PLAN_WARPS) * ipt * g.tpw * R > 65536 ||
                       smem2(ipt, g.tpw) > kSmemBudget))
        --ipt;
    while (g.tpw > 1 && (static_cast<int64_t>(moe::PLAN_WARPS) * ipt * g.tpw * R > 65536 ||
                         smem2(ipt, g.tpw) > kSmemBudget))
        g.tpw >>= 1;
    g.ipt = static_cast<int>(ipt);
    g.tile_tokens = moe::PLAN_WARPS * g.ipt * g.tpw;
    g.T = static_cast<int>((static_cast<int64_t>(N) + g.tile_tokens - 1) / g.tile_tokens);
    g.C = E + R + 2;
    return g;
}

size_t ws_bytes(const Geom& g) {
    size_t b = sizeof(moe::WsHeader);
    b += sizeof(uint64_t) * static_cast<size_t>(g.T) * g.C + 8;  // + 16-byte alignment of tile_prefix
    b += sizeof(int32_t) * static_cast<size_t>(g.T) * g.C;
    return (b + 15) / 16 * 16;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// N = 0 is a valid, empty batch.
int check_sizes(int N, int E, int K, int R) {
    if (N < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E || R < 1 || R > 128 || E % R != 0)
        return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(N) * K >= (int64_t(1) << 30)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

namespace {

constexpr int kMaxClusterTiles = 16;

size_t cluster_smem(const Geom& g, int E, int R);

// Tiles for the one-launch cluster path: as few iterations per warp as keep
// the tile count within 16.  False when the plan needs more tiles or when
// the tile's is_token_in_rank rows exceed 64 KB.
bool cluster_geometry(int N, int E, int K, int R, Geom* g) {
    g->tpw = 32 / K;
    const int64_t per_tile_iter = static_cast<int64_t>(moe::PLAN_WARPS) * g->tpw;  // tokens
    const int64_t tiles1 = (static_cast<int64_t>(N) + per_tile_iter - 1) / per_tile_iter;
    const int64_t ipt = (tiles1 + kMaxClusterTiles - 1) / kMaxClusterTiles;
    if (ipt > moe::PLAN_IPT_MAX) return false;
    g->ipt = static_cast<int>(ipt < 1 ? 1 : ipt);
    g->tile_tokens = moe::PLAN_WARPS * g->ipt * g->tpw;
    if (static_cast<int64_t>(g->tile_tokens) * R > 65536) return false;
    g->T = static_cast<int>((static_cast<int64_t>(N) + g->tile_tokens - 1) / g->tile_tokens);
    g->C = E + R + 2;
    return g->T >= 1 && g->T <= kMaxClusterTiles && cluster_smem(*g, E, R) <= 220 * 1024;
}

size_t cluster_smem(const Geom& g, int E, int R) {
    const size_t ints = static_cast<size_t>(2 * moe::PLAN_WARPS * 32) * g.ipt + static_cast<size_t>(moe::PLAN_WARPS) * E +
                        2 * static_cast<size_t>(g.C) + E + 2 * static_cast<size_t>(E + R + 2) + 4;  // + alignment
    return sizeof(int32_t) * ints + (static_cast<size_t>(g.tile_tokens) * R + 15) / 16 * 16;
}

cudaLaunchConfig_t cluster_config(int T, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T);
    cfg.blockDim = dim3(moe::PLAN_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = T;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cfg;
}

// Whether a cluster of T CTAs of `kernel` with this much dynamic shared
// memory fits the GPU (cached per device, kernel, size and shared memory).
template <typename Kernel>
bool cluster_launchable(Kernel kernel, int T, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int, size_t>, bool> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const auto key = std::make_tuple(dev, reinterpret_cast<const void*>(kernel), T, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config(T, smem, nullptr, attr, false);
    int n = 0;
    const bool ok = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n >= 1;
    if (!ok) cudaGetLastError();  // clear a sticky-free query error
    cache[key] = ok;
    return ok;
}

template <typename Kernel, typename... Args>
int launch_cluster(Kernel kernel, int T, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config(T, smem, stream, attr, moe_host::pdl_enabled());
    return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---- small-E path geometry: 32 warps per CTA, the fewest warp steps
// (1, 2, 4, 8) that keep the tiles within 16 (one cluster).
bool small_geometry(int N, int E, int K, int R, Geom* g) {
    if (E > moe::SMALL_MAX || R > moe::SMALL_MAX) return false;
    g->tpw = 32 / K;
    g->C = E + R + 2;
    for (int ipt : {1, 2, 4, 8}) {
        g->ipt = ipt;
        g->tile_tokens = moe::PLAN_WARPS * ipt * g->tpw;
        const int64_t T = (static_cast<int64_t>(N) + g->tile_tokens - 1) / g->tile_tokens;
        if (T <= kMaxClusterTiles) {
            g->T = static_cast<int>(T);
            return true;
        }
    }
    return false;
}

// Fused route + plan kernels (E <= 8: the logits of a token in two float4;
// K <= 2 or K <= 8 winners per lane).
template <int KM, typename F>
auto with_fused_kernel_k(int ipt, F&& f) {
    switch (ipt) {
        case 1: return f(moe::plan_small_kernel<1, 3, moe::RouteSource<8, KM>>, moe::RouteSource<8, KM>{});
        case 2: return f(moe::plan_small_kernel<2, 3, moe::RouteSource<8, KM>>, moe::RouteSource<8, KM>{});
        case 4: return f(moe::plan_small_kernel<4, 3, moe::RouteSource<8, KM>>, moe::RouteSource<8, KM>{});
        default: return f(moe::plan_small_kernel<8, 3, moe::RouteSource<8, KM>>, moe::RouteSource<8, KM>{});
    }
}
template <typename F>
auto with_fused_kernel(int ipt, int K, F&& f) {
    return K <= 2 ? with_fused_kernel_k<2>(ipt, f) : with_fused_kernel_k<8>(ipt, f);
}

// ---- medium-E path geometry: 32 < E <= 256, R <= 32, 32 warps per CTA,
// the fewest warp steps (1, 2, 4) that keep the tiles within 16.
bool medium_geometry(int N, int E, int K, int R, Geom* g) {
    if (E <= moe::SMALL_MAX || E > 256 || R > moe::SMALL_MAX) return false;
    g->tpw = 32 / K;
    g->C = E + R + 2;
    for (int ipt : {1, 2, 4}) {
        g->ipt = ipt;
        g->tile_tokens = moe::PLAN_WARPS * ipt * g->tpw;
        const int64_t T = (static_cast<int64_t>(N) + g->tile_tokens - 1) / g->tile_tokens;
        if (T <= kMaxClusterTiles) {
            g->T = static_cast<int>(T);
            return true;
        }
    }
    return false;
}

size_t medium_smem(const Geom& g, int E) {
    return sizeof(int32_t) * (static_cast<size_t>(moe::PLAN_WARPS) * E + 4 * 256 + 16 * static_cast<size_t>(g.C) +
                              3 * static_cast<size_t>(E) + 2 * static_cast<size_t>(moe::PLAN_WARPS) * 32 * g.ipt);
}

// EW = 4 when E <= 128, else 8.
template <typename F>
auto with_medium_kernel(int ipt, int E, F&& f) {
    if (E <= 128) {
        switch (ipt) {
            case 1: return f(moe::plan_medium_kernel<1, 4>);
            case 2: return f(moe::plan_medium_kernel<2, 4>);
            default: return f(moe::plan_medium_kernel<4, 4>);
        }
    }
    switch (ipt) {
        case 1: return f(moe::plan_medium_kernel<1, 8>);
        case 2: return f(moe::plan_medium_kernel<2, 8>);
        default: return f(moe::plan_medium_kernel<4, 8>);
    }
}

// NB = 3 when E <= 8 (so R <= 8), else 5.
template <typename F>
auto with_small_kernel(int ipt, int E, F&& f) {
    if (E <= 8) {
        switch (ipt) {
            case 1: return f(moe::plan_small_kernel<1, 3, moe::TopkSource>);
            case 2: return f(moe::plan_small_kernel<2, 3, moe::TopkSource>);
            case 4: return f(moe::plan_small_kernel<4, 3, moe::TopkSource>);
            default: return f(moe::plan_small_kernel<8, 3, moe::TopkSource>);
        }
    }
    switch (ipt) {
        case 1: return f(moe::plan_small_kernel<1, 5, moe::TopkSource>);
        case 2: return f(moe::plan_small_kernel<2, 5, moe::TopkSource>);
        case 4: return f(moe::plan_small_kernel<4, 5, moe::TopkSource>);
        default: return f(moe::plan_small_kernel<8, 5, moe::TopkSource>);
    }
}

// ---- grid path geometry: one warp iteration per tile with the fewest warps
// (8, 16, 32) that keep the tiles within 152, else 32 warps and as many
// iterations as needed (at most PLAN_IPT_MAX).  A function of the sizes
// alone, like the workspace it implies; whether the tiles can all be
// resident at once is checked per device at launch.
constexpr int kGridMaxTiles = 152;

size_t grid_smem(const Geom& g, int warps, int E, int R) {
    const size_t ints = static_cast<size_t>(2 * warps * 32) * g.ipt + static_cast<size_t>(warps) * E +
                        3 * static_cast<size_t>(g.C) + 2 * static_cast<size_t>(E + R + 2) + 4;  // + alignment
    return sizeof(int32_t) * ints + (static_cast<size_t>(g.tile_tokens) * R + 15) / 16 * 16;
}

bool grid_geometry(int N, int E, int K, int R, Geom* g, int* warps) {
    g->tpw = 32 / K;
    int w = 0;
    int64_t ipt = 1;
    for (int cand : {8, 16, 32}) {
        const int64_t tt = static_cast<int64_t>(cand) * g->tpw;
        if ((static_cast<int64_t>(N) + tt - 1) / tt <= kGridMaxTiles) {
            w = cand;
            break;
        }
    }
    if (w == 0) {
        w = 32;
        const int64_t per = static_cast<int64_t>(w) * g->tpw * kGridMaxTiles;
        ipt = (static_cast<int64_t>(N) + per - 1) / per;
        if (ipt > moe::PLAN_IPT_MAX) return false;
    }
    g->ipt = static_cast<int>(ipt);
    g->tile_tokens = static_cast<int>(w * ipt * g->tpw);
    g->T = static_cast<int>((static_cast<int64_t>(N) + g->tile_tokens - 1) / g->tile_tokens);
    g->C = E + R + 2;
    *warps = w;
    if (static_cast<int64_t>(g->tile_tokens) * R > 65536) return false;
    return g->T >= 1 && g->T <= kGridMaxTiles && grid_smem(*g, w, E, R) <= 220 * 1024;
}

// header, then flags u64[T], then counts i32[C][T]
size_t grid_ws_bytes(const Geom& g) {
    const size_t b = sizeof(moe::WsHeader) + sizeof(uint64_t) * static_cast<size_t>(g.T) + 8 +
                     sizeof(int32_t) * static_cast<size_t>((g.T + 3) & ~3) * g.C;
    return (b + 15) / 16 * 16;
}

// Workspace for every path the sizes allow.
size_t plan_ws_bytes(int N, int E, int K, int R) {
    if (N == 0) return sizeof(moe::WsHeader);  // the empty plan reads no workspace
    size_t b = ws_bytes(plan_geometry(N, E, K, R));
    Geom gg;
    int w = 0;
    if (grid_geometry(N, E, K, R, &gg, &w)) b = std::max(b, grid_ws_bytes(gg));
    return b;
}

template <int W>
int grid_occupancy(size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, moe::plan_grid_kernel<W>, W * 32, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Whether all T CTAs can be resident at once (cached per device and shape).
bool grid_launchable(int warps, int T, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t>, bool> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const auto key = std::make_tuple(dev, warps, T, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const int per_sm = warps == 8 ? grid_occupancy<8>(smem) : warps == 16 ? grid_occupancy<16>(smem)
                                                                          : grid_occupancy<32>(smem);
    const bool ok = static_cast<int64_t>(per_sm) * moe_host::num_sms() >= T;
    cache[key] = ok;
    return ok;
}

int launch_grid(int warps, const PlanArgs& a, size_t smem, cudaStream_t stream) {
    const dim3 grid(a.T), block(warps * 32);
    if (warps == 8) return moe_host::launch(moe::plan_grid_kernel<8>, grid, block, smem, stream, a);
    if (warps == 16) return moe_host::launch(moe::plan_grid_kernel<16>, grid, block, smem, stream, a);
    return moe_host::launch(moe::plan_grid_kernel<32>, grid, block, smem, stream, a);
}

// Dynamic shared memory limits of every plan kernel, once per device.
int ensure_kernel_attributes() {
    static std::mutex mu;
    static std::map<int, cudaError_t> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(dev);
    if (it == done.end()) {
        const int big = 220 * 1024;  // the geometries keep every plan kernel within this
        const cudaError_t errs[] = {
            cudaFuncSetAttribute(moe::plan_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_grid_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_grid_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_grid_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_small_kernel<1, 3, moe::TopkSource>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<2, 3, moe::TopkSource>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<4, 3, moe::TopkSource>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<8, 3, moe::TopkSource>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<1, 5, moe::TopkSource>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<2, 5, moe::TopkSource>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<4, 5, moe::TopkSource>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<8, 5, moe::TopkSource>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<1, 3, moe::RouteSource<8, 2>>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<1, 3, moe::RouteSource<8, 8>>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<2, 3, moe::RouteSource<8, 2>>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<2, 3, moe::RouteSource<8, 8>>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<4, 3, moe::RouteSource<8, 2>>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<4, 3, moe::RouteSource<8, 8>>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<8, 3, moe::RouteSource<8, 2>>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_small_kernel<8, 3, moe::RouteSource<8, 8>>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_medium_kernel<1, 4>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_medium_kernel<2, 4>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_medium_kernel<4, 4>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_medium_kernel<1, 8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_medium_kernel<2, 8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_medium_kernel<4, 8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
            cudaFuncSetAttribute(moe::plan_medium_kernel<1, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_medium_kernel<2, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_medium_kernel<4, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_medium_kernel<1, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_medium_kernel<2, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, big),
            cudaFuncSetAttribute(moe::plan_medium_kernel<4, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, big)};
        cudaError_t first = cudaSuccess;
        for (cudaError_t e : errs)
            if (first == cudaSuccess) first = e;
        it = done.emplace(dev, first).first;
    }
    return it->second == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Which path a plan of these sizes takes on the current device.  Default
// order: the small-E cluster kernel, the medium-E cluster kernel, then the
// two-launch look-back plan.  MOE_PLAN_PATH=small|medium|cluster|grid|lookback
// forces a path where the sizes allow it (the look-back plan otherwise).
enum PlanPath { PATH_SMALL = 0, PATH_CLUSTER = 1, PATH_GRID = 2, PATH_LOOKBACK = 3, PATH_MEDIUM = 4 };

struct PathChoice {
    int path;
    Geom g;
    int warps;
    size_t smem;
};

PathChoice choose_path(int N, int E, int K, int R) {
    const char* env = std::getenv("MOE_PLAN_PATH");
    const std::string want = env != nullptr ? env : "auto";
    const bool any = want == "auto";
    Geom g;
    int w = 0;
    if ((any || want == "small") && small_geometry(N, E, K, R, &g)) {
        const bool ok = with_small_kernel(g.ipt, E, [&](auto kern) { return cluster_launchable(kern, g.T, 0); });
        if (ok) return PathChoice{PATH_SMALL, g, moe::PLAN_WARPS, 0};
    }
    if ((any || want == "medium") && medium_geometry(N, E, K, R, &g)) {
        const size_t smem = medium_smem(g, E);
        const bool ok = with_medium_kernel(g.ipt, E, [&](auto kern) { return cluster_launchable(kern, g.T, smem); });
        if (ok) return PathChoice{PATH_MEDIUM, g, moe::PLAN_WARPS, smem};
    }
    if (want == "cluster" && cluster_geometry(N, E, K, R, &g)) {
        const size_t smem = cluster_smem(g, E, R);
        if (cluster_launchable(moe::plan_cluster_kernel, g.T, smem)) return PathChoice{PATH_CLUSTER, g, moe::PLAN_WARPS, smem};
    }
    if (want == "grid" && grid_geometry(N, E, K, R, &g, &w)) {
        const size_t smem = grid_smem(g, w, E, R);
        if (grid_launchable(w, g.T, smem)) return PathChoice{PATH_GRID, g, w, smem};
    }
    return PathChoice{PATH_LOOKBACK, plan_geometry(N, E, K, R), moe::PLAN_WARPS, 0};
}

}  // namespace

extern "C" MOE_API int64_t moe_plan_capacity_rows(int N, int E, int K, int alignment) {
    if (N < 0 || E < 1 || K < 1 || alignment < 1) return -1;
    return static_cast<int64_t>(N) * K + static_cast<int64_t>(E) * (alignment - 1);
}

extern "C" MOE_API size_t moe_plan_workspace_size(int N, int E, int K, int R) {
    if (check_sizes(N, E, K, R) != MOE_OK) return 0;
    return plan_ws_bytes(N, E, K, R);
}

extern "C" MOE_API int moe_plan_launch_count(int N, int E, int K, int R) {
    if (check_sizes(N, E, K, R) != MOE_OK) return -1;
    if (N == 0) return 1;  // plan_empty_kernel
    if (ensure_kernel_attributes() != MOE_OK) return -1;
    return choose_path(N, E, K, R).path == PATH_LOOKBACK ? 2 : 1;
}

extern "C" MOE_API int moe_plan_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (workspace == nullptr || workspace_bytes < sizeof(moe::WsHeader) || !aligned(workspace, 16))
        return MOE_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

namespace {

// Host checks of a plan call, and its argument block without the tile
// geometry and the workspace layout (those depend on the path).
int plan_args(const int32_t* topk_idx, int N, int E, int K, int R, int alignment, void* workspace,
              size_t workspace_bytes, const MoePlanOut* out, PlanArgs* a) {
    int rc = check_sizes(N, E, K, R);
    if (rc != MOE_OK) return rc;
    if (alignment < 1 || topk_idx == nullptr || workspace == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
    const int64_t p_cap = moe_plan_capacity_rows(N, E, K, alignment);
    if (p_cap >= (int64_t(1) << 31) - 1) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {out->tokens_per_expert, out->cu_seqlens, out->zero_fill_ranges, out->pairs_per_rank,
                          out->tokens_per_rank,   out->rank_prefix, out->rank_slot_offsets, out->dst,
                          out->src_of_slot,       out->dup_groups,  out->dup_loffs,     out->dup_counts,
                          out->status,            topk_idx};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned(p, 4)) return MOE_ERR_INVALID_ARG;
    if (out->is_token_in_rank == nullptr || !aligned(workspace, 16)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < plan_ws_bytes(N, E, K, R)) return MOE_ERR_CAPACITY;
    rc = ensure_kernel_attributes();
    if (rc != MOE_OK) return rc;

    a->topk = topk_idx;
    a->out = *out;
    a->hdr = static_cast<moe::WsHeader*>(workspace);
    a->flags = nullptr;
    a->tile_prefix = nullptr;
    a->N = N;
    a->E = E;
    a->K = K;
    a->R = R;
    a->epn = E / R;
    a->epn_magic = (uint64_t(1) << 32) / static_cast<uint64_t>(a->epn) + 1;
    a->alignment = alignment;
    a->p_cap = p_cap;
    a->skip_tile = moe_host::skip_tile();
    a->timeout_ns = moe_host::timeout_ns();
    return MOE_OK;
}

}  // namespace

namespace {

// The plan of an empty batch (N = 0): one small launch that writes the
// E- and R-sized outputs and marks the capacity rows unused.  topk_idx, the
// workspace and the N-sized arrays (dst, is_token_in_rank, dup_groups,
// dup_loffs) are not touched and may be null; src_of_slot may be null when
// the capacity E * (alignment - 1) is zero.
int plan_empty(int E, int K, int R, int alignment, const MoePlanOut* out, cudaStream_t stream) {
    if (check_sizes(0, E, K, R) != MOE_OK || alignment < 1 || out == nullptr) return MOE_ERR_INVALID_ARG;
    const int64_t p_cap = moe_plan_capacity_rows(0, E, K, alignment);
    if (p_cap < 0 || p_cap >= (int64_t(1) << 31) - 1) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {out->tokens_per_expert, out->cu_seqlens,        out->zero_fill_ranges, out->pairs_per_rank,
                          out->tokens_per_rank,   out->rank_prefix,       out->rank_slot_offsets, out->dup_counts,
                          out->status};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned(p, 4)) return MOE_ERR_INVALID_ARG;
    if (p_cap > 0 && (out->src_of_slot == nullptr || !aligned(out->src_of_slot, 4))) return MOE_ERR_INVALID_ARG;
    int64_t blocks = (p_cap + 255) / 256;
    const int64_t cap = static_cast<int64_t>(moe_host::num_sms()) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return moe_host::launch(moe::plan_empty_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, *out, E,
                            R, p_cap);
}

}  // namespace

extern "C" MOE_API int moe_plan(const int32_t* topk_idx, int N, int E, int K, int R, int alignment,
                                void* workspace, size_t workspace_bytes, const MoePlanOut* out,
                                cudaStream_t stream) {
    if (N == 0) return plan_empty(E, K, R, alignment, out, stream);
    PlanArgs a;
    int rc = plan_args(topk_idx, N, E, K, R, alignment, workspace, workspace_bytes, out, &a);
    if (rc != MOE_OK) return rc;
    const PathChoice pc = choose_path(N, E, K, R);
    const Geom& g = pc.g;
    a.flags = reinterpret_cast<uint64_t*>(static_cast<char*>(workspace) + sizeof(moe::WsHeader));
    {
        // the grid path reads its counts with 16-byte loads: start them on a
        // 16-byte boundary (the workspace itself is 16-byte aligned)
        const uintptr_t p = reinterpret_cast<uintptr_t>(a.flags + static_cast<size_t>(g.T) * (pc.path == PATH_GRID ? 1 : g.C));
        a.tile_prefix = reinterpret_cast<int32_t*>((p + 15) & ~static_cast<uintptr_t>(15));
    }
    a.tpw = g.tpw;
    a.ipt = g.ipt;
    a.tile_tokens = g.tile_tokens;
    a.T = g.T;
    a.C = g.C;

    // ---- one launch: a thread-block cluster of up to 16 tiles, E, R <= 32
    if (pc.path == PATH_SMALL)
        return with_small_kernel(g.ipt, E, [&](auto kern) { return launch_cluster(kern, a.T, 0, stream, a, moe::TopkSource{}); });
    // ---- one launch: a thread-block cluster of up to 16 tiles, 32 < E <= 256, R <= 32
    if (pc.path == PATH_MEDIUM)
        return with_medium_kernel(g.ipt, E, [&](auto kern) { return launch_cluster(kern, a.T, pc.smem, stream, a); });
    // ---- one launch: a thread-block cluster of up to 16 tiles, any E
    if (pc.path == PATH_CLUSTER) return launch_cluster(moe::plan_cluster_kernel, a.T, pc.smem, stream, a);
    // ---- one launch over the whole GPU, all tiles resident at once
    if (pc.path == PATH_GRID) return launch_grid(pc.warps, a, pc.smem, stream);
    // ---- two launches: decoupled look-back over tiles, then the scatter
    const size_t smem1 = sizeof(int32_t) * (static_cast<size_t>(g.C) + 2 * (E + R + 2) + 2);
    const size_t smem2 = sizeof(int32_t) * (static_cast<size_t>(moe::PLAN_WARPS + 1) * E +
                                            static_cast<size_t>(2 * moe::PLAN_WARPS * 32) * g.ipt + 4) +
                         (static_cast<size_t>(g.tile_tokens) * R + 15) / 16 * 16;
    rc = moe_host::launch(moe::plan_count_kernel, dim3(g.T), dim3(moe::PLAN_THREADS), smem1, stream, a);
    if (rc != MOE_OK) return rc;
    return moe_host::launch(moe::plan_scatter_kernel, dim3(g.T), dim3(moe::PLAN_THREADS), smem2, stream, a);
}

// ---------------------------------------------------------------- fused route + plan
extern "C" MOE_API int moe_route_plan_fused(int N, int E, int K, int R, int n_group) {
    if (check_sizes(N, E, K, R) != MOE_OK) return -1;
    if (N == 0) return 0;  // nothing to route: the plan alone runs
    if (ensure_kernel_attributes() != MOE_OK) return -1;
    // opt-in: on GB300 the fused launch measured slower than the two calls
    // (routing on the plan's 16 SMs costs what the routing kernel costs on
    // all of them, whose launch the dependent-launch chain already hides)
    if (env_int("MOE_ROUTE_PLAN_FUSED", 0) != 1) return 0;
    const char* env = std::getenv("MOE_PLAN_PATH");
    if (env != nullptr && std::string(env) != "auto" && std::string(env) != "small") return 0;
    Geom g;
    if (n_group != 1 || E > 8 || E % 4 != 0 || K > moe::FUSED_KMAX || (K & (K - 1)) != 0 ||
        !small_geometry(N, E, K, R, &g))
        return 0;
    return with_fused_kernel(g.ipt, K, [&](auto kern, auto) { return cluster_launchable(kern, g.T, 0); }) ? 1 : 0;
}

extern "C" MOE_API int moe_route_plan(const float* logits, const float* bias, int N, int E, int K, int scoring,
                                      int renormalize, int n_group, int topk_group, float routed_scaling,
                                      int32_t* topk_idx, float* topk_w, int R, int alignment, void* workspace,
                                      size_t workspace_bytes, const MoePlanOut* out, cudaStream_t stream) {
    const int fused = moe_route_plan_fused(N, E, K, R, n_group);
    if (fused < 0) return MOE_ERR_INVALID_ARG;
    if (fused == 0) {  // two calls: the routing kernel, then the plan
        const int rc = moe_route_topk(logits, bias, N, E, K, scoring, renormalize, n_group, topk_group,
                                      routed_scaling, topk_idx, topk_w, stream);
        if (rc != MOE_OK) return rc;
        return moe_plan(topk_idx, N, E, K, R, alignment, workspace, workspace_bytes, out, stream);
    }
    moe::RouteArgs ra;
    int rc = moe_host::route_args(logits, bias, N, E, K, scoring, renormalize, n_group, topk_group, routed_scaling,
                                  topk_idx, topk_w, &ra);
    if (rc != MOE_OK) return rc;
    PlanArgs a;
    rc = plan_args(topk_idx, N, E, K, R, alignment, workspace, workspace_bytes, out, &a);
    if (rc != MOE_OK) return rc;
    Geom g;
    small_geometry(N, E, K, R, &g);
    a.tpw = g.tpw;
    a.ipt = g.ipt;
    a.tile_tokens = g.tile_tokens;
    a.T = g.T;
    a.C = g.C;
    return with_fused_kernel(g.ipt, K, [&](auto kern, auto src) {
        src.r = ra;
        return launch_cluster(kern, a.T, 0, stream, a, src);
    });
}

// ---------------------------------------------------------------- no-allocation variant
// Scratch for moe_plan_no_alloc: a fixed device array in this library's
// module, so the call needs no caller workspace and allocates nothing.
// Every GPU that loads the library holds these bytes until the process
// exits.  Host code must not use the symbol itself as a device address; the
// address comes from cudaGetSymbolAddress with the device current.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_plan_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on
// every call: a device reset (or a torn-down primary context) reloads the
// module, and the array may then sit at a new address with unknown contents.
// Whenever the address differs from the one last seen on this device (the
// first call included), the array is zeroed on `stream` before use (the
// plan's call counter and look-back flags start from zero).
int scratch_for_current_device(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] != p) {
        if (cudaMemsetAsync(p, 0, kNoAllocScratchBytes, stream) != cudaSuccess) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = p;
    return MOE_OK;
}

}  // namespace

extern "C" MOE_API int moe_plan_no_alloc(const int32_t* topk_idx, int N, int E, int K, int R, int alignment,
                                         const MoePlanOut* out, cudaStream_t stream) {
    int rc = check_sizes(N, E, K, R);
    if (rc != MOE_OK) return rc;
    if (alignment < 1) return MOE_ERR_INVALID_ARG;
    const size_t need = plan_ws_bytes(N, E, K, R);
    if (need > kNoAllocScratchBytes) return MOE_ERR_CAPACITY;
    void* ws = nullptr;
    rc = scratch_for_current_device(stream, &ws);
    if (rc != MOE_OK) return rc;
    return moe_plan(topk_idx, N, E, K, R, alignment, ws, kNoAllocScratchBytes, out, stream);
}
