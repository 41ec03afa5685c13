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
// rank_prefix, tokens in order inside a block).  A CTA per rank counts its
// column of is_token_in_rank in contiguous token chunks, scans the chunk
// counts, then writes the slots and the channel prefixes.
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

constexpr int LAYOUT_THREADS = 1024;

struct RankLayoutArgs {
    const uint8_t* itr;
    const int32_t* rank_prefix;
    int32_t* status;
    int32_t* channel_prefix_matrix;
    int32_t* token_rank_slot;
    int N, R, C;
};

__global__ void __launch_bounds__(LAYOUT_THREADS) rank_layout_kernel(const RankLayoutArgs a) {
    __shared__ int32_t s_warp[LAYOUT_THREADS / 32 + 1];
    __shared__ int32_t s_base[LAYOUT_THREADS];  // tokens of rank r before each chunk
    __shared__ int32_t s_total;
    pdl_wait();
    pdl_trigger();
    if (ld_volatile_s32(a.status) != 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    const int R = a.R;
    const int64_t N = a.N;
    const int64_t chunk = (N + LAYOUT_THREADS - 1) / LAYOUT_THREADS;
    const int64_t b = min(N, tid * chunk), e = min(N, b + chunk);
    int32_t cnt = 0;
    for (int64_t s = b; s < e; ++s) cnt += a.itr[s * R + r] ? 1 : 0;
    // block exclusive scan of the chunk counts
    int32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(FULL_MASK, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int32_t v = s_warp[lane];
        int32_t w = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(FULL_MASK, w, off);
            if (lane >= off) w += y;
        }
        s_warp[lane] = w - v;
    }
    __syncthreads();
    const int32_t excl = s_warp[warp] + incl - cnt;
    s_base[tid] = excl;
    if (tid == LAYOUT_THREADS - 1) s_total = excl + cnt;
    // slots of this chunk
    const int32_t rank_base = __ldg(a.rank_prefix + r);
    int32_t run = rank_base + excl;
    for (int64_t s = b; s < e; ++s) {
        const bool in = a.itr[s * R + r] != 0;
        a.token_rank_slot[s * R + r] = in ? run : -1;
        run += in ? 1 : 0;
    }
    __syncthreads();
    // channel c ends at token end_c: tokens of rank r before it
    const int64_t q = (N + a.C - 1) / a.C;
    for (int c = tid; c < a.C; c += LAYOUT_THREADS) {
        const int64_t end = min(N, (static_cast<int64_t>(c) + 1) * q);
        int32_t v = s_total;
        if (end < N) {
            const int64_t owner = end / chunk;  // chunk holding token `end` (< LAYOUT_THREADS)
            v = s_base[owner];
            for (int64_t s = owner * chunk; s < end; ++s) v += a.itr[s * R + r] ? 1 : 0;
        }
        a.channel_prefix_matrix[static_cast<size_t>(r) * a.C + c] = v;
    }
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

extern "C" MOE_API int moe_rank_layout(const MoePlanOut* plan, int N, int R, int num_channels,
                                       int32_t* channel_prefix_matrix, int32_t* token_rank_slot,
                                       cudaStream_t stream) {
    if (plan == nullptr || plan->is_token_in_rank == nullptr || plan->rank_prefix == nullptr ||
        plan->status == nullptr || channel_prefix_matrix == nullptr || token_rank_slot == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (N < 1 || R < 1 || R > 128 || num_channels < 1 || static_cast<int64_t>(N) * R >= (int64_t(1) << 31))
        return MOE_ERR_INVALID_ARG;
    moe::RankLayoutArgs a;
    a.itr = plan->is_token_in_rank;
    a.rank_prefix = plan->rank_prefix;
    a.status = plan->status;
    a.channel_prefix_matrix = channel_prefix_matrix;
    a.token_rank_slot = token_rank_slot;
    a.N = N;
    a.R = R;
    a.C = num_channels;
    return moe_host::launch(moe::rank_layout_kernel, dim3(R), dim3(moe::LAYOUT_THREADS), 0, stream, a);
}
