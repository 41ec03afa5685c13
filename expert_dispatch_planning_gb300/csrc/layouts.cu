// layouts.cu -- layouts derived from a plan, for the consumers of the
// permuted buffer and of a deduplicated per-rank buffer.
//
// moe_tile_map: the grouped-GEMM tile map of TensorRT-LLM RoutingKernel.cuh
// (routingPermutation: CtaIdxXyToBatchIdx, CtaIdxXyToMnLimit,
// PermutedIdxSize, NumNonExitingCtas) over the plan's padded expert rows:
// with tiles of `alignment` rows every expert's rows start on a tile, so
// tile t belongs to the expert whose rows contain row t*alignment (binary
// search over cu_seqlens) and ends at min((t+1)*alignment, cu[e] + count).
// A thread per tile; tiles past the padded total hold -1.
//
// moe_rank_layout: DeepEP csrc/kernels/intranode.cu, notify_dispatch's
// channel prefix matrix (per destination rank, tokens of each channel that
// go to it, inclusive prefix over channels) and the per-(token, rank) slot
// of a buffer that holds each token once per rank it needs (rank blocks at
// rank_prefix, tokens in order inside a block), in two launches over token
// tiles (below).
#include "moe_common.cuh"

namespace moe {

struct TileMapArgs {
    const int32_t* cu;
    const int32_t* counts;
    int32_t* status;
    int32_t* tile_expert;
    int32_t* tile_row_limit;
    int32_t* sizes;
    int E, alignment;
    int64_t max_tiles;
};

__global__ void __launch_bounds__(256) tile_map_kernel(const TileMapArgs a) {
    pdl_wait();
    pdl_trigger();
    if (ld_volatile_s32(a.status) != 0) return;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= a.max_tiles) return;
    const int32_t P = __ldg(a.cu + a.E);
    const int64_t num_tiles = P / a.alignment;
    if (t == 0) {
        a.sizes[0] = static_cast<int32_t>(num_tiles);
        a.sizes[1] = P;
    }
    if (t >= num_tiles) {
        a.tile_expert[t] = -1;
        a.tile_row_limit[t] = -1;
        return;
    }
    const int64_t row = t * a.alignment;
    int lo = 0, hi = a.E;  // last expert e with cu[e] <= row: upper bound - 1
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.cu + mid) <= row)
            lo = mid + 1;
        else
            hi = mid;
    }
    const int e = lo - 1;
    const int64_t end = static_cast<int64_t>(__ldg(a.cu + e)) + __ldg(a.counts + e);
    a.tile_expert[t] = e;
    a.tile_row_limit[t] = static_cast<int32_t>(min(row + a.alignment, end));
}

// ---- rank layout: two launches over tiles of TT tokens (TT a multiple of 32)
//
// Launch 1, a CTA per tile: for every 32-token chunk and rank, the bit mask
// of the chunk's tokens that go to the rank (a warp ballot per rank over its
// 32 rows), and the tile's token count per rank.  Launch 2, a CTA per tile:
// the tile's base per rank (sum of earlier tiles' counts), a running base per
// chunk, then every (token, rank) slot from its chunk base plus the popcount
// of the mask bits below it (one thread per output element, so the int32
// rows are written contiguously), and the channel prefixes whose channel end
// falls in the tile.  Workspace: masks [T][TT/32][R], counts [T][R].
constexpr int LAYOUT_THREADS = 256;
constexpr int LAYOUT_WARPS = LAYOUT_THREADS / 32;

struct RankLayoutArgs {
    const uint8_t* itr;
    const int32_t* rank_prefix;
    int32_t* status;
    int32_t* channel_prefix_matrix;
    int32_t* token_rank_slot;
    uint32_t* masks;  // [T][TT/32][R]
    int32_t* counts;  // [T][R]
    int N, R, C, TT, T;
};

__global__ void __launch_bounds__(LAYOUT_THREADS) rank_layout_mask_kernel(const RankLayoutArgs a) {
    extern __shared__ int32_t s_cnt[];  // [R]
    pdl_wait();
    pdl_trigger();
    if (ld_volatile_s32(a.status) != 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = a.R, tile = blockIdx.x;
    const int chunks = a.TT / 32;
    const int64_t s0 = static_cast<int64_t>(tile) * a.TT;
    for (int r = tid; r < R; r += LAYOUT_THREADS) s_cnt[r] = 0;
    __syncthreads();
    uint32_t* tmask = a.masks + static_cast<size_t>(tile) * chunks * R;
    // rows as 4-byte words when every row starts on a 4-byte boundary
    const bool words = (R % 4) == 0 && (reinterpret_cast<uintptr_t>(a.itr) % 4) == 0;
    for (int c = warp; c < chunks; c += LAYOUT_WARPS) {
        const int64_t s = s0 + 32 * c + lane;
        const bool valid = s < a.N;
        const uint8_t* row = a.itr + (valid ? s : 0) * R;
        uint32_t w[32];  // the row's bytes (R <= 128), every load in flight at once
#pragma unroll
        for (int q = 0; q < 32; ++q) w[q] = 0u;
        if (words) {
#pragma unroll
            for (int q = 0; q < 32; ++q)
                if (4 * q < R && valid) w[q] = __ldg(reinterpret_cast<const uint32_t*>(row) + q);
        } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (4 * q + u < R && valid) w[q] |= static_cast<uint32_t>(__ldg(row + 4 * q + u)) << (8 * u);
            }
        }
        uint32_t mine[4] = {0u, 0u, 0u, 0u};  // masks of ranks lane, lane + 32, ...
#pragma unroll
        for (int q = 0; q < 32; ++q) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = 4 * q + u;
                if (r < R) {
                    const uint32_t m = __ballot_sync(FULL_MASK, ((w[q] >> (8 * u)) & 0xffu) != 0u);
                    if (lane == (r & 31)) mine[r >> 5] = m;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int r = 32 * q + lane;
            if (r < R) {
                tmask[c * R + r] = mine[q];
                if (mine[q] != 0u) atomicAdd(&s_cnt[r], __popc(mine[q]));
            }
        }
    }
    __syncthreads();
    for (int r = tid; r < R; r += LAYOUT_THREADS) a.counts[static_cast<size_t>(tile) * R + r] = s_cnt[r];
}

__global__ void __launch_bounds__(LAYOUT_THREADS) rank_layout_slot_kernel(const RankLayoutArgs a) {
    extern __shared__ int32_t s_dyn[];
    const int R = a.R, tile = blockIdx.x;
    const int chunks = a.TT / 32;
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_dyn);   // [chunks][R]
    int32_t* s_cbase = s_dyn + chunks * R;                    // [chunks + 1][R]: tokens before each chunk
    int32_t* s_part = s_cbase + (chunks + 1) * R;             // [LAYOUT_WARPS][R] partial tile sums
    int32_t* s_rp = s_part + LAYOUT_WARPS * R;                // [R] rank_prefix
    pdl_wait();
    pdl_trigger();
    if (ld_volatile_s32(a.status) != 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t s0 = static_cast<int64_t>(tile) * a.TT;
    const int64_t s1 = min(static_cast<int64_t>(a.N), s0 + a.TT);

    // tokens of earlier tiles, per rank: warp w sums tiles w, w + 8, ...
    // (eight loads in flight per lane)
    for (int r0 = 0; r0 < R; r0 += 32) {
        const int r = r0 + lane;
        int32_t v = 0;
        if (r < R) {
            int t = warp;
            for (; t + 7 * LAYOUT_WARPS < tile; t += 8 * LAYOUT_WARPS) {
                int32_t x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] = __ldg(a.counts + static_cast<size_t>(t + u * LAYOUT_WARPS) * R + r);
#pragma unroll
                for (int u = 0; u < 8; ++u) v += x[u];
            }
            for (; t < tile; t += LAYOUT_WARPS) v += __ldg(a.counts + static_cast<size_t>(t) * R + r);
            s_part[warp * R + r] = v;
        }
    }
    const uint32_t* tmask = a.masks + static_cast<size_t>(tile) * chunks * R;
    for (int i = tid; i < chunks * R; i += LAYOUT_THREADS) s_mask[i] = __ldg(tmask + i);
    for (int r = tid; r < R; r += LAYOUT_THREADS) s_rp[r] = __ldg(a.rank_prefix + r);
    __syncthreads();
    for (int r = tid; r < R; r += LAYOUT_THREADS) {
        int32_t run = 0;
#pragma unroll
        for (int w = 0; w < LAYOUT_WARPS; ++w) run += s_part[w * R + r];
        for (int c = 0; c < chunks; ++c) {
            s_cbase[c * R + r] = run;
            run += __popc(s_mask[c * R + r]);
        }
        s_cbase[chunks * R + r] = run;  // tokens before the tile's end
    }
    __syncthreads();

    // slots: a warp per token row (R >= 32: lanes over ranks) or 32 / R rows
    // per warp (R < 32: lane = (row, rank)); rows are written contiguously
    const int ntok = static_cast<int>(s1 - s0);
    int32_t* out = a.token_rank_slot + s0 * R;
    const int rpp = R >= 32 ? 1 : 32 / R;
    const int ro = R >= 32 ? 0 : lane / R;
    const int r_first = R >= 32 ? lane : lane - ro * R;
    const int r_step = R >= 32 ? 32 : R;
    if (ro < rpp) {
        for (int sl = warp * rpp + ro; sl < ntok; sl += LAYOUT_WARPS * rpp) {
            const int c = sl >> 5, b = sl & 31;
            const uint32_t below = (1u << b) - 1u;
            for (int r = r_first; r < R; r += r_step) {
                const uint32_t m = s_mask[c * R + r];
                out[static_cast<int64_t>(sl) * R + r] = ((m >> b) & 1u) ? s_rp[r] + s_cbase[c * R + r] + __popc(m & below) : -1;
            }
        }
    }

    // channel c ends at token e_c = min((c + 1) q, N): tokens of rank r
    // before e_c, written by the tile holding token e_c (the last tile also
    // takes e_c = N); this tile's channels are c_lo..c_hi
    const int64_t q = (static_cast<int64_t>(a.N) + a.C - 1) / a.C;
    const bool last = tile == a.T - 1;
    const int64_t c_lo = max(int64_t(0), (s0 + q - 1) / q - 1);
    const int64_t c_hi = last ? a.C - 1 : min(static_cast<int64_t>(a.C) - 1, (s1 - 1) / q - 1);
    for (int64_t c = c_lo + warp; c <= c_hi; c += LAYOUT_WARPS) {
        const int64_t ec = min(static_cast<int64_t>(a.N), (c + 1) * q);
        for (int r = lane; r < R; r += 32) {
            int32_t v;
            if (ec >= s0 && ec < s1) {
                const int sl = static_cast<int>(ec - s0), cc = sl >> 5, b = sl & 31;
                v = s_cbase[cc * R + r] + __popc(s_mask[cc * R + r] & ((1u << b) - 1u));
            } else if (last && ec == s1) {
                v = s_cbase[chunks * R + r];
            } else {
                continue;
            }
            a.channel_prefix_matrix[static_cast<size_t>(r) * a.C + c] = v;
        }
    }
}

// An empty batch (N = 0): every channel prefix is zero.  Writes nothing
// after a failed plan, like the other layout kernels.
__global__ void __launch_bounds__(LAYOUT_THREADS) rank_layout_empty_kernel(int32_t* cpm, const int32_t* status,
                                                                         int64_t n) {
    pdl_wait();
    pdl_trigger();
    if (ld_volatile_s32(status) != 0) return;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) cpm[i] = 0;
}

}  // namespace moe

extern "C" MOE_API int moe_tile_map(const MoePlanOut* plan, int E, int alignment, int32_t* tile_expert,
                                    int32_t* tile_row_limit, int64_t max_tiles, int32_t* sizes,
                                    cudaStream_t stream) {
    if (plan == nullptr || plan->cu_seqlens == nullptr || plan->tokens_per_expert == nullptr ||
        plan->status == nullptr || tile_expert == nullptr || tile_row_limit == nullptr || sizes == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || alignment < 1 || max_tiles < 1 || max_tiles >= (int64_t(1) << 31))
        return MOE_ERR_INVALID_ARG;
    moe::TileMapArgs a;
    a.cu = plan->cu_seqlens;
    a.counts = plan->tokens_per_expert;
    a.status = plan->status;
    a.tile_expert = tile_expert;
    a.tile_row_limit = tile_row_limit;
    a.sizes = sizes;
    a.E = E;
    a.alignment = alignment;
    a.max_tiles = max_tiles;
    const unsigned blocks = static_cast<unsigned>((max_tiles + 255) / 256);
    return moe_host::launch(moe::tile_map_kernel, dim3(blocks), dim3(256), 0, stream, a);
}

namespace {

// Tiles of TT tokens: about 256 tiles, TT a multiple of 32, at most 4096
// (chunk, rank) masks per tile (the slot kernel keeps two such arrays in
// shared memory, under 48 KB in all).
struct LayoutGeom {
    int TT, T;
};
LayoutGeom layout_geom(int N, int R) {
    int64_t tt = (static_cast<int64_t>(N) + 255) / 256;
    tt = ((tt + 31) / 32) * 32;
    const int64_t cap = (4096 / R) * 32;
    if (tt > cap) tt = cap;
    if (tt < 32) tt = 32;
    LayoutGeom g;
    g.TT = static_cast<int>(tt);
    g.T = static_cast<int>((N + tt - 1) / tt);
    return g;
}

size_t layout_ws_bytes(int N, int R) {
    const LayoutGeom g = layout_geom(N, R);
    const size_t masks = static_cast<size_t>(g.T) * (g.TT / 32) * R * sizeof(uint32_t);
    return ((masks + 255) / 256) * 256 + static_cast<size_t>(g.T) * R * sizeof(int32_t);
}

}  // namespace

extern "C" MOE_API size_t moe_rank_layout_workspace_size(int N, int R) {
    if (N == 0 && R >= 1 && R <= 128) return 256;  // an empty batch reads no workspace
    if (N < 1 || R < 1 || R > 128 || static_cast<int64_t>(N) * R >= (int64_t(1) << 31)) return 0;
    return layout_ws_bytes(N, R);
}

extern "C" MOE_API int moe_rank_layout(const MoePlanOut* plan, int N, int R, int num_channels, void* workspace,
                                       size_t workspace_bytes, int32_t* channel_prefix_matrix,
                                       int32_t* token_rank_slot, cudaStream_t stream) {
    if (plan == nullptr || plan->status == nullptr || channel_prefix_matrix == nullptr) return MOE_ERR_INVALID_ARG;
    if (N == 0) {
        // an empty batch: no channel holds a token; is_token_in_rank,
        // token_rank_slot and the workspace are not touched (NULL allowed)
        if (R < 1 || R > 128 || num_channels < 1) return MOE_ERR_INVALID_ARG;
        const int64_t n = static_cast<int64_t>(R) * num_channels;
        int64_t blocks = (n + moe::LAYOUT_THREADS - 1) / moe::LAYOUT_THREADS;
        const int64_t cap = static_cast<int64_t>(moe_host::num_sms()) * 4;
        if (blocks > cap) blocks = cap;
        return moe_host::launch(moe::rank_layout_empty_kernel, dim3(static_cast<unsigned>(blocks)),
                                dim3(moe::LAYOUT_THREADS), 0, stream, channel_prefix_matrix, plan->status, n);
    }
    if (plan->is_token_in_rank == nullptr || plan->rank_prefix == nullptr || token_rank_slot == nullptr ||
        workspace == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (N < 1 || R < 1 || R > 128 || num_channels < 1 || static_cast<int64_t>(N) * R >= (int64_t(1) << 31))
        return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < layout_ws_bytes(N, R)) return MOE_ERR_CAPACITY;
    const LayoutGeom g = layout_geom(N, R);
    const size_t mask_bytes = static_cast<size_t>(g.T) * (g.TT / 32) * R * sizeof(uint32_t);
    moe::RankLayoutArgs a;
    a.itr = plan->is_token_in_rank;
    a.rank_prefix = plan->rank_prefix;
    a.status = plan->status;
    a.channel_prefix_matrix = channel_prefix_matrix;
    a.token_rank_slot = token_rank_slot;
    a.masks = static_cast<uint32_t*>(workspace);
    a.counts = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + ((mask_bytes + 255) / 256) * 256);
    a.N = N;
    a.R = R;
    a.C = num_channels;
    a.TT = g.TT;
    a.T = g.T;
    const int chunks = g.TT / 32;
    int rc = moe_host::launch(moe::rank_layout_mask_kernel, dim3(g.T), dim3(moe::LAYOUT_THREADS),
                              sizeof(int32_t) * R, stream, a);
    if (rc != MOE_OK) return rc;
    const size_t smem = sizeof(int32_t) * (static_cast<size_t>(chunks) * R + (chunks + 1) * R +
                                           static_cast<size_t>(moe::LAYOUT_WARPS) * R + R);
    return moe_host::launch(moe::rank_layout_slot_kernel, dim3(g.T), dim3(moe::LAYOUT_THREADS), smem, stream, a);
}
