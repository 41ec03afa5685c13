/*
 * moe_dispatch.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts routing
 * and dispatch-planning library.
 *
 * One GPU, one CUDA stream per call.  "Ranks" are logical partitions of the
 * experts computed on this GPU: rank r owns experts [r*E/R, (r+1)*E/R).
 *
 * Conventions shared by every entry point
 *   - Pointers marked (device) point to device memory owned by the caller;
 *     the library allocates nothing and keeps no pointer after a call.
 *   - Buffers must not alias one another unless a function says so.
 *   - bf16 tensors are passed as their 16-bit patterns (uint16_t).
 *   - A call validates its arguments on the host, enqueues its kernels on
 *     `stream` and returns without synchronising.  Arguments are checked
 *     before any CUDA call, so an invalid call has no effect.
 *   - Return value: MOE_OK or one of the MOE_ERR_* codes below.  Errors that
 *     only the device can see (an expert id outside [0, E), a bounded wait
 *     that ran out) are recorded in the plan's device status word and read
 *     with moe_get_status().
 *   - Flat pair index f = s*K + k for token s and its k-th expert.
 *   - N = 0 (a batch with no tokens) is valid everywhere N is taken.
 *     Pointers to arrays that then have no elements may be NULL.
 *
 * Sources (page title and section):
 *   MoonEP moonep/planning.py -- PlanningKernel (histogram, per-expert
 *     prefix over blocks, stable scatter, per-rank cu_seqlens and
 *     zero_fill_ranges, dst, duplicate canonicalisation, src_info), the
 *     MoonEPCommPlan record, allocate_planning_outputs / launch_planning
 *     (caller-allocated outputs written in place), _check_dedup_encoding_bounds.
 *   TensorRT-LLM trtllmGenKernels/blockScaleMoe/RoutingKernel.cuh --
 *     calcSoftmax, sigmoid_accurate, routingIndicesHistogramKernel /
 *     routingIndicesOffsetsKernel (expanded -> permuted index).
 *   DeepEP csrc/kernels/intranode.cu -- notify_dispatch (rank prefix
 *     matrix, aligned per-expert receive counts, is_token_in_rank),
 *     dispatch (hidden-row copy), combine (fp32 accumulation, bf16 store),
 *     host-side argument assertions.
 */
#ifndef MOE_DISPATCH_H
#define MOE_DISPATCH_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* ---------------------------------------------------------------- status */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1      /* a size, pointer or option is out of range      */
#define MOE_ERR_UNSUPPORTED 2      /* a valid combination this library does not run  */
#define MOE_ERR_CAPACITY 3         /* a caller buffer is smaller than required       */
#define MOE_ERR_CUDA 4             /* a CUDA runtime call or kernel launch failed    */
#define MOE_ERR_DEVICE_TIMEOUT 5   /* (device) a bounded wait ran out                */
#define MOE_ERR_DEVICE_INDEX 6     /* (device) an expert id or slot out of range     */
#define MOE_ERR_WORKSPACE 7        /* (device) plan workspace not initialised        */
#define MOE_ERR_DEVICE_CAPACITY 8  /* (device) a rank's groups exceed its row budget */

#define MOE_SCORING_SOFTMAX 0
#define MOE_SCORING_SIGMOID 1

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(int code);

/* ---------------------------------------------------------------- router */
/*
 * Router top-K (TensorRT-LLM calcSoftmax / sigmoid_accurate; tie rule of
 * MoonEP warp_argmax_min_idx).
 *
 *   logits        (device) float32[N][E], row-major, 16-byte aligned.
 *   bias          (device) float32[E] correction bias or NULL; sigmoid only.
 *   scoring       MOE_SCORING_SOFTMAX: the selection key is the logit;
 *                 MOE_SCORING_SIGMOID: key = sigmoid(logit) + bias, with
 *                 sigmoid evaluated by one fixed fp32 sequence
 *                 (1/(1+e^-x) for x >= 0, e^x/(1+e^x) otherwise; e^t by
 *                 Cody-Waite reduction with ln2 split 16+24 bits and the
 *                 degree-7 Taylor polynomial in Horner form with fused
 *                 multiply-adds; scaling by two exact powers of two).
 *   n_group,      group-limited selection (sigmoid only): experts form
 *   topk_group    n_group contiguous groups (n_group <= 32, E % n_group
 *                 == 0); a group scores the fp32 sum of its two largest
 *                 keys; the topk_group best groups are kept and top-K runs
 *                 over their experts.  n_group = 1 disables it.
 *   K             1 <= K <= 32, K <= E (and <= topk_group*E/n_group).
 *   renormalize   softmax: weights are the softmax over the K selected
 *                 logits (1) or over all E (0).  sigmoid: w_k = s_k / sum
 *                 of the K selected scores (1) or s_k (0).  Scores are
 *                 unbiased.  All weights are multiplied by routed_scaling.
 *   topk_idx      (device) int32[N][K] out: descending key, equal keys in
 *                 ascending expert index.
 *   topk_w        (device) float32[N][K] out, within 1e-6 relative of the
 *                 exact value.
 * 0 <= N (N = 0 launches nothing), 1 <= E <= 1024, E % 4 == 0 for the
 * vector path (any E works).
 * NaN logits are outside the contract (their position in the order is
 * unspecified).
 *
 * From 16384 tokens on, with E = 32*G (G = 4, 8 or 16) and K <= 8, sigmoid
 * scores with n_group 1 or G and K <= G, and renormalised softmax scores
 * without groups, take a faster kernel with the same output bit for bit
 * (launched in plain stream order): it chooses candidates by
 * approximate keys (sigmoid: hardware ex2/rcp approximations, within 2^-20
 * of the fixed sigmoid for every fp32 input; softmax: the logit with its 5
 * low bits replaced by the expert's position), checks that the
 * chosen top-K set and kept groups are separated from the rest by more
 * than twice the keys' error bound, evaluates the fixed sigmoid only for
 * the winners, and routes any token that fails a check (and every token
 * when a bias is not finite or exceeds 2^20) with the exact kernel's code,
 * a warp per token after the block's other tokens (a block takes at most
 * 512 tokens; very large N launches several waves of blocks).
 * MOE_ROUTE_PATH=exact in the environment keeps every call on the exact
 * kernel; MOE_ROUTE_PATH=fast takes the fast one at any token count.
 */
MOE_API int moe_route_topk(const float* logits, const float* bias, int N, int E, int K,
                           int scoring, int renormalize, int n_group, int topk_group,
                           float routed_scaling, int32_t* topk_idx, float* topk_w,
                           cudaStream_t stream);

/* ---------------------------------------------------------------- plan */
/*
 * Caller-owned plan outputs (MoonEP MoonEPCommPlan, DeepEP notify_dispatch
 * outputs, in their single-GPU form).  Every pointer is device memory,
 * 4-byte aligned (is_token_in_rank may have any alignment; at 16 bytes its
 * rows are written with vector stores).  P denotes the padded row total
 * cu_seqlens[E]; P_cap = moe_plan_capacity_rows(...).
 */
typedef struct MoePlanOut {
    int32_t* tokens_per_expert;  /* [E]     pairs routed to each expert                    */
    int32_t* cu_seqlens;         /* [E+1]   0, then running sum of padded counts; padded
                                    = round_up(count, alignment) if count > 0 else 0      */
    int32_t* zero_fill_ranges;   /* [E][2]  (cu[e]+count, padded-count) if positive, else
                                    (0, 0)                                                */
    int32_t* pairs_per_rank;     /* [R]     pairs routed to each rank's experts           */
    int32_t* tokens_per_rank;    /* [R]     tokens with at least one pair on the rank     */
    int32_t* rank_prefix;        /* [R+1]   exclusive prefix of tokens_per_rank           */
    int32_t* rank_slot_offsets;  /* [R+1]   cu_seqlens[r*E/R]: first row of each rank     */
    uint8_t* is_token_in_rank;   /* [N][R]  1 if token s has a pair on rank r            */
    int32_t* dst;                /* [N][K]  raw slot (row of the permuted buffer) of the
                                    pair; -slot-1 when an earlier k of the same token
                                    already reached that rank (a duplicate)               */
    int32_t* src_of_slot;        /* [P_cap] flat pair index f of each row, -1 for padding
                                    and unused rows                                       */
    int32_t* dup_groups;         /* [N*(K/2)][3] (primary slot, dup_begin, dup_count) for
                                    each (token, rank) holding >= 2 pairs, in (token,
                                    first k) order                                        */
    int32_t* dup_loffs;          /* [N*(K-1)] duplicate slots, group after group, k order */
    int32_t* dup_counts;         /* [2]     (number of groups, number of duplicates)     */
    int32_t* status;             /* [4]     device status: [0] first error code (0 = ok),
                                    [1] detail.  Zero it before first use; read and
                                    cleared by moe_get_status.                            */
} MoePlanOut;

/* Rows the permuted buffer needs: N*K + E*(alignment-1) (N >= 0).  -1 on bad
 * input. */
MOE_API int64_t moe_plan_capacity_rows(int N, int E, int K, int alignment);

/* Bytes of device workspace moe_plan needs for these sizes (0 on bad input). */
MOE_API size_t moe_plan_workspace_size(int N, int E, int K, int R);

/*
 * Kernel launches moe_plan makes for these sizes on the current device: 1
 * when R <= 32, E <= 256 and the plan fits one thread-block cluster of up to
 * 16 tiles (one tile = 32 warps x 1, 2, 4 or 8 steps x floor(32/K) tokens;
 * at most 4 steps when E > 32) that the GPU can co-schedule, else 2
 * (decoupled look-back, then the scatter); 1 for N = 0 (the empty plan).
 * -1 on bad sizes.  The
 * environment variable MOE_PLAN_PATH=small|medium|cluster|grid|lookback
 * forces a path where the sizes allow it (cluster: a one-launch cluster
 * plan for any E; grid: one launch of up to 152 co-resident tiles); every
 * path produces the identical plan.
 */
MOE_API int moe_plan_launch_count(int N, int E, int K, int R);

/*
 * Prepare a workspace for its first use (enqueues a memset on `stream`).
 * A workspace carries a call counter between calls, so it must be
 * initialised once after allocation; afterwards any number of moe_plan
 * calls (of any sizes it fits) may use it, one at a time.
 */
MOE_API int moe_plan_workspace_init(void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream);

/*
 * Dispatch plan (MoonEP PlanningKernel; TensorRT-LLM histogram / offsets
 * kernels; DeepEP notify_dispatch).
 *
 *   topk_idx   (device) int32[N][K] expert ids in [0, E).
 *   R          logical ranks, E % R == 0, R <= 128 (MoonEP's rank-bitset
 *              bound); alignment >= 1 rows per expert.
 *   workspace  (device) >= moe_plan_workspace_size(N, E, K, R) bytes,
 *              16-byte aligned, initialised once (moe_plan_workspace_init).
 *              Two plans in flight at once must not share a workspace.
 *   out        host struct of device pointers (see MoePlanOut).
 *
 * Slots are canonical: within each expert, pairs keep ascending flat index
 * (MoonEP's stable scatter order), so the plan is a pure function of
 * topk_idx.  N = 0 plans an empty batch in one small launch: every count,
 * offset and prefix is 0, zero_fill_ranges are (0, 0), src_of_slot is -1 on
 * all E*(alignment-1) rows; topk_idx, the workspace and the N-sized arrays
 * are not touched (NULL allowed), nor src_of_slot when alignment is 1.
 * Checked here: N >= 0, 1 <= K <= 32, K <= E <= 1024,
 * E % R == 0, R <= 128, N*K < 2^30, P_cap < 2^31.  Recorded in the status
 * word by the device: MOE_ERR_DEVICE_INDEX (an expert id outside [0, E)),
 * MOE_ERR_WORKSPACE (a workspace that was never initialised),
 * MOE_ERR_DEVICE_TIMEOUT (a wait on another tile ran out: 1 s); after an
 * error the plan's outputs are unspecified and moe_permute / moe_combine
 * with this plan write nothing.
 */
MOE_API int moe_plan(const int32_t* topk_idx, int N, int E, int K, int R, int alignment,
                     void* workspace, size_t workspace_bytes, const MoePlanOut* out,
                     cudaStream_t stream);

/*
 * moe_plan without a workspace argument, for callers that cannot allocate
 * device memory: code embedded in a host framework that owns every device
 * buffer and hands out only inputs and outputs, or latency-critical callers
 * that must not run cudaMalloc/cudaFree (which can synchronise the whole
 * device) and have no spare buffer to lend.  The sources have no counterpart:
 * MoonEP and TensorRT-LLM both take caller- or framework-allocated scratch.
 *
 * The plan's scratch lives in a fixed 1 MiB device array inside this library
 * (every GPU that loads the library holds it until the process exits).  Sizes
 * whose moe_plan_workspace_size() exceeds 1 MiB return MOE_ERR_CAPACITY; the
 * five reference workloads (up to N = 65536, E = 256, K = 8, R = 64) need
 * under 0.6 MiB.  The call allocates nothing and runs the same kernels as
 * moe_plan, so its outputs are identical.
 *
 * Every call looks up the array's device address on the current device.
 * The first call on a device, and any call that finds the array at a new
 * address (after a device reset reloaded the library's module), zeroes it
 * with a memset enqueued on `stream`: make the first call on each device
 * before any stream capture.  All calls on a device share the one array and
 * it keeps the previous call's state, so calls that may overlap on the GPU (different
 * streams without ordering between them) race and give wrong plans: order
 * them on one stream or use moe_plan with separate workspaces.
 */
MOE_API int moe_plan_no_alloc(const int32_t* topk_idx, int N, int E, int K, int R, int alignment,
                              const MoePlanOut* out, cudaStream_t stream);

/*
 * Plan reuse (MoonEP MoonEPCommPlan.clone; DeepEP's cached dispatch reuses
 * a plan instead of planning again).  A plan is caller-owned and stays valid
 * for any number of moe_permute / moe_combine calls while its buffers live;
 * this copies plan `src` into the buffers of `dst` (same N, E, K, R,
 * alignment), one asynchronous device-to-device copy per array on `stream`.
 */
MOE_API int moe_plan_copy(const MoePlanOut* src, const MoePlanOut* dst, int N, int E, int K, int R,
                          int alignment, cudaStream_t stream);

/* ---------------------------------------------------------------- balanced plan */
/*
 * Capacity-balanced logical-rank plan with redundant experts (MoonEP
 * moonep/planning.py, PlanningKernel: the balancing matrix z, the
 * allocation of each owner's expert pairs to other ranks, the top-B remote
 * expert selection, per-rank padded groups, and dst by the allocation
 * prefix in the rank*NvS + loff encoding), in its one-GPU form: a single
 * source rank, so the per-expert token totals are the plain plan's counts.
 * All arrays are caller-owned device memory, int32, 4-byte aligned.
 */
typedef struct MoeBalancedPlanOut {
    int32_t* z;                /* [R][R]  pairs moved from rank i to rank j              */
    int32_t* alloc;            /* [R][E]  pairs of expert e handled by rank r            */
    int32_t* alloc_cumsum;     /* [E][R]  inclusive prefix of alloc over ranks           */
    int32_t* experts_to_copy;  /* [R][B]  redundant experts per rank, -1 for none        */
    int32_t* remote_stats;     /* [R][2]  (remote experts with pairs, times picked)      */
    int32_t* rank_cu_seqlens;  /* [R][E+B] padded group ends, rank-local                 */
    int32_t* rank_zero_fill;   /* [R][E+B][2] (start, count) of each group's padding     */
    int32_t* expert_offsets;   /* [R][E]  first row of expert e's group on rank r (0 if
                                  the rank holds none of its pairs)                      */
    int32_t* dst;              /* [N][K]  r*NvS + row on rank r; -value-1 for a later
                                  pair of the token on an already-used rank              */
} MoeBalancedPlanOut;

/*
 * plan         a plan built by moe_plan for the same topk_idx (its counts,
 *              cu_seqlens and dst give each pair's position among its
 *              expert's pairs); its status word receives device errors.
 * capacity     CAP: pairs a rank should hold before balancing moves pairs to
 *              ranks below it (MoonEP's NvS_capacity).
 * B            redundant-expert slots per rank, 0 <= B <= 64.
 * token_padding  rows each group is padded to (>= 1).
 * NvS          rows per rank in the dst encoding; R*NvS < 2^31.  A rank whose
 *              groups need more rows sets MOE_ERR_DEVICE_CAPACITY.
 * Three launches on `stream` after the plain plan (two when N = 0: nothing
 * to balance, every matrix zero, every experts_to_copy entry -1; topk_idx
 * and the dst arrays may then be NULL); no workspace.
 */
MOE_API int moe_plan_balanced(const MoePlanOut* plan, const int32_t* topk_idx, int N, int E, int K, int R,
                              int token_padding, int32_t capacity, int B, int32_t NvS,
                              const MoeBalancedPlanOut* out, cudaStream_t stream);

/* ---------------------------------------------------------------- layouts */
/*
 * Grouped-GEMM tile map (TensorRT-LLM RoutingKernel.cuh, routingPermutation:
 * CtaIdxXyToBatchIdx, CtaIdxXyToMnLimit, NumNonExitingCtas,
 * PermutedIdxSize) over a plan's permuted buffer, with tiles of `alignment`
 * rows (the plan's alignment, so every expert starts on a tile).
 *   tile_expert     (device) int32[max_tiles]: expert of tile t (global id),
 *                   -1 from num_tiles on.
 *   tile_row_limit  (device) int32[max_tiles]: one past the tile's last real
 *                   row, min((t+1)*alignment, cu[e] + count[e]); -1 past the end.
 *   sizes           (device) int32[2]: (num_tiles, padded rows P).
 * max_tiles >= P_cap / alignment covers every plan of these sizes.
 */
MOE_API int moe_tile_map(const MoePlanOut* plan, int E, int alignment, int32_t* tile_expert,
                         int32_t* tile_row_limit, int64_t max_tiles, int32_t* sizes, cudaStream_t stream);

/*
 * Rank layout (DeepEP csrc/kernels/intranode.cu, notify_dispatch).
 *   channel_prefix_matrix  (device) int32[R][num_channels]: tokens of channels
 *                   0..c that go to rank r; channel c covers tokens
 *                   [c*q, (c+1)*q), q = ceil(N / num_channels).
 *   token_rank_slot (device) int32[N][R]: the row of token s in a buffer that
 *                   holds each token once per rank it needs, ranks' blocks
 *                   at rank_prefix[r], tokens in order; -1 if s does not go
 *                   to r.
 *   workspace       (device) moe_rank_layout_workspace_size(N, R) bytes,
 *                   256-byte aligned, caller-owned; needs no initialisation
 *                   (every call rewrites what it reads).  Calls sharing a
 *                   workspace must not overlap on the GPU.
 * Reads the plan's is_token_in_rank and rank_prefix.  R <= 128.  Two kernel
 * launches.  MOE_ERR_CAPACITY if the workspace is too small.  N = 0: one
 * launch that zeroes channel_prefix_matrix; is_token_in_rank,
 * token_rank_slot and the workspace are not touched (NULL allowed).
 */
MOE_API size_t moe_rank_layout_workspace_size(int N, int R);
MOE_API int moe_rank_layout(const MoePlanOut* plan, int N, int R, int num_channels, void* workspace,
                            size_t workspace_bytes, int32_t* channel_prefix_matrix, int32_t* token_rank_slot,
                            cudaStream_t stream);

/*
 * Routing and the dispatch plan in one call (TensorRT-LLM RoutingKernel.cuh,
 * routingPermutation, the single-cluster variant that routes and permutes in
 * one launch below a token count; MoonEP's plan outputs).  Results are those
 * of moe_route_topk followed by moe_plan with the same arguments, bit for
 * bit (the kernel runs the router's own arithmetic).  One launch when
 * moe_route_plan_fused() returns 1 for the sizes, else exactly those two
 * calls.  Arguments: as for moe_route_topk and moe_plan (topk_idx and
 * topk_w are written in both cases; the workspace is moe_plan's).
 */
MOE_API int moe_route_plan(const float* logits, const float* bias, int N, int E, int K, int scoring,
                           int renormalize, int n_group, int topk_group, float routed_scaling,
                           int32_t* topk_idx, float* topk_w, int R, int alignment, void* workspace,
                           size_t workspace_bytes, const MoePlanOut* out, cudaStream_t stream);

/*
 * 1 when moe_route_plan runs as one launch for these sizes on the current
 * device: the environment variable MOE_ROUTE_PLAN_FUSED=1 is set, there is no
 * group limit (n_group == 1), E <= 8 with E % 4 == 0, K is a power of two
 * <= 8, R <= 32 and the plan fits one thread-block cluster of up to 16 CTAs;
 * 0 when it makes the two calls (the default: the one launch measured slower
 * on GB300, since it routes on the cluster's 16 SMs while the routing kernel
 * uses all of them); -1 on bad sizes.
 */
MOE_API int moe_route_plan_fused(int N, int E, int K, int R, int n_group);

/* ---------------------------------------------------------------- rows */
/* moe_permute flags. */
#define MOE_PERMUTE_EARLY_X 1  /* see moe_permute */

/*
 * Permute (DeepEP dispatch's hidden-row copy, MoonEP dst / zero_fill_ranges):
 *   permuted[raw slot(f)] = x[f / K] for every pair, primaries and
 *   duplicates alike; rows inside the zero-fill ranges are written +0.0;
 *   rows at or beyond cu_seqlens[E] are left untouched.
 *   x         (device) bf16[N][H], 16-byte aligned; H % 8 == 0.
 *   permuted  (device) bf16[P_cap][H], 16-byte aligned, must not alias x.
 *   plan      the plan built by moe_plan for the same N, E, K, alignment
 *             (uses dst, zero_fill_ranges, status).
 *   flags     0, or MOE_PERMUTE_EARLY_X: the kernel starts loading x rows
 *             before the kernel enqueued just before it on `stream` has
 *             finished (it waits for that kernel before reading the plan).
 *             Allowed only when that kernel does not write x -- as when
 *             moe_permute directly follows the moe_plan call that built
 *             `plan` and x was produced before it; never when x comes from
 *             the kernel right before (a plan reused for new hidden states).
 * If the plan's status holds an error the call writes nothing.  Other
 * flag bits: MOE_ERR_INVALID_ARG.
 */
MOE_API int moe_permute(const uint16_t* x, int N, int H, int K, int E, int alignment,
                        const MoePlanOut* plan, uint16_t* permuted, int flags, cudaStream_t stream);

/*
 * Weighted combine (DeepEP combine's fp32 accumulation and bf16 store):
 *   out[s][h] = bf16_rne(acc), acc = 0, then for k = 0..K-1
 *       acc = fmaf(topk_w[s][k], float(y[raw slot(s,k)][h]), acc).
 *   y       (device) bf16[P_cap][H] expert outputs in permuted order.
 *   topk_w  (device) float32[N][K].
 *   out     (device) bf16[N][H]; must not alias y.
 *   plan    uses dst and status.
 */
MOE_API int moe_combine(const uint16_t* y, const float* topk_w, int N, int K, int H, int E,
                        int alignment, const MoePlanOut* plan, uint16_t* out,
                        cudaStream_t stream);

/* ---------------------------------------------------------------- status */
/*
 * Synchronise `stream`, copy the plan's device status to *device_status
 * (MOE_OK or a MOE_ERR_DEVICE_* / MOE_ERR_WORKSPACE code) and clear it.
 * Returns MOE_ERR_CUDA if the synchronisation or copy fails.
 */
MOE_API int moe_get_status(const MoePlanOut* plan, int32_t* device_status, cudaStream_t stream);

/*
 * Self-check of the fast router's error bound: writes to *max_abs_err
 * (device, one float) the largest |approximate sigmoid - fixed sigmoid|
 * over every non-NaN fp32 input (2^32 evaluations, a few ms).  The fast
 * router's margins assume 2^-20.  No counterpart on the pages.
 */
MOE_API int moe_debug_route_sigmoid_error(float* max_abs_err, cudaStream_t stream);

/*
 * Test hook for the bounded-wait path: while skip_tile >= 0, the planning
 * kernel's tile `skip_tile` never publishes its counts, so later tiles wait
 * until `timeout_ns` runs out and report MOE_ERR_DEVICE_TIMEOUT.  Pass
 * (-1, 0) to restore the defaults (no skipped tile, 1 s limit).
 */
MOE_API int moe_debug_set_plan_fault(int skip_tile, int64_t timeout_ns);

#ifdef __cplusplus
}
#endif
#endif /* MOE_DISPATCH_H */
