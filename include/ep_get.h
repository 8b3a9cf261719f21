/*
 * ep_get.h -- C ABI of the GB300 MoE token dispatch / combine library
 * (libep_get.so, CUDA kernels for sm_103a).
 *
 * The hot path is routing layout -> dispatch -> combine for R expert-parallel
 * ranks that are logical partitions of ONE GPU's memory: a "rank" is a
 * contiguous block of E/R experts and a contiguous block of rows in the
 * receive buffer.  There is no traffic between GPUs.
 *
 * Sources (page title, then section or code fragment):
 *  - "DeepEP Symmetric Memory" architecture analysis, section 6.1: the
 *    dispatch launch carries per-rank and per-expert prefix sums of receive
 *    counts, a destination slot index per token, expert_alignment, FP8 scale
 *    factor packs and strides, topk_idx and topk_weights;
 *    section 7.3: the host learns the receive count per rank and per local
 *    expert after dispatch; section 9.2: dispatch(x, topk_idx, topk_weights,
 *    num_experts) returns recv_x, recv_topk_idx, recv_topk_weights and a
 *    handle, and combine(x, handle, topk_weights) returns the combined rows.
 *  - "DeepEP V2 ElasticBuffer architecture", TokenLayout fragment: a received
 *    token carries its hidden row, its scale factors, its top-k indices
 *    (4 bytes each), its top-k weights (4 bytes each) and its source token
 *    index (4 bytes); limits fragment: at most 1024 ranks, 2048 experts and
 *    256 experts per rank.
 *
 * Conventions shared by every entry point:
 *  - All array arguments are DEVICE pointers owned by the caller; they must be
 *    16-byte aligned.  The library allocates nothing and keeps no state
 *    between calls other than per-device kernel attributes, the built-in
 *    scratch array of ep_get_layout_static_scratch and a process-wide call
 *    counter that numbers the rows-ready tags of ep_layout_and_dispatch.
 *  - Every call is asynchronous on `cuda_stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  The caller orders streams.
 *  - Errors a host check can see (null or misaligned pointers, sizes out of
 *    range, unsupported shapes) are returned before anything is launched.
 *  - Errors only the device can see are OR-ed into the caller's device word
 *    `*d_status` (int32, zero it before the first call); the offending entry
 *    or row is skipped and every other result is still correct.  Read it after
 *    the stream has synchronised.  Nothing ever traps.
 *  - A return of EP_ERR_CUDA means a launch failed; cudaGetLastError() has
 *    the CUDA error.
 *  - Logging: with the environment variable EP_GET_DEBUG set to anything but
 *    "0" when the library is first used, every call writes one line on
 *    stderr ("[ep_get] <entry point>: <shapes and options>"), every host check
 *    that rejects a call one more (the status and the check's source line),
 *    and every kernel launch one (kernel, grid, block, dynamic shared memory,
 *    cluster size).  Unset, nothing is written.  The counterpart of the
 *    EP_BUFFER_DEBUG switch ("DeepEP Symmetric Memory", App. B).
 *
 * Notation: T tokens (all source ranks together), H hidden channels, K top-k
 * slots per token, E experts, R ranks, E_l = E/R experts per rank; expert e
 * lives on rank e / E_l.  Token t's source rank is t / (T/R) when R divides
 * T.  n(t) is the number of distinct ranks among t's valid experts and
 * N = sum_t n(t) is the number of received rows.
 */
#ifndef EP_GET_H
#define EP_GET_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status bits (returned and/or OR-ed into *d_status). */
typedef int32_t ep_status_t;
#define EP_OK                0
#define EP_ERR_INVALID_ARG   1   /* host: bad pointer, size or alignment        */
#define EP_ERR_UNSUPPORTED   2   /* host: shape beyond the limits below         */
#define EP_ERR_INVALID_INDEX 4   /* device: a topk_idx entry outside [-1, E)    */
#define EP_ERR_CAPACITY      8   /* device: a row index >= the receive capacity */
#define EP_ERR_TIMEOUT       16  /* device: a bounded wait gave up              */
#define EP_ERR_CUDA          32  /* host: a CUDA launch failed                  */
/* device, bounds-checked build only (compiled with EP_GET_CHECKED=1): an
 * index failed the check against its array's extent, or a dst_row /
 * expanded_row / node_row entry was below -1; the access was skipped,
 * nothing traps.  The product build never sets it (it reads an entry below
 * -1 as "absent", like -1). */
#define EP_ERR_OUT_OF_BOUNDS 64

/* Payload types of the receive buffer. */
#define EP_BF16      0
#define EP_FP8_E4M3  1

/* Limits ("DeepEP V2 ElasticBuffer architecture", limits fragment), plus the
 * top-k width this library supports. */
#define EP_MAX_RANKS            1024
#define EP_MAX_EXPERTS          2048
#define EP_MAX_EXPERTS_PER_RANK 256
#define EP_MAX_TOPK             32

/*
 * The routing layout: the dispatch "handle".  All members are device pointers
 * owned by the caller.  Filled by ep_get_layout, read by ep_dispatch and
 * ep_combine; one layout serves any number of dispatch/combine calls (the
 * pages' cached mode).
 */
typedef struct ep_layout {
    int32_t* num_tokens_per_rank;   /* [R]   tokens received by each rank                 */
    int32_t* num_tokens_per_node;   /* [R/ranks_per_node] tokens per node group, or NULL  */
    int32_t* num_tokens_per_expert; /* [E]   valid top-k entries naming each expert       */
    uint8_t* is_token_in_rank;      /* [T,R] 1 if any valid expert of t is on r, else 0   */
    int32_t* rank_offset;           /* [R+1] exclusive prefix of num_tokens_per_rank;
                                             rank_offset[R] = N                          */
    int32_t* expert_offset;         /* [E+1] exclusive prefix of num_tokens_per_expert,
                                             each rounded up to expert_alignment         */
    int32_t* dst_row;               /* [T,R] receive row of (t, r) or -1; rows of rank r
                                             are rank_offset[r] + 0, 1, ... in ascending t */
    int32_t* src_dst_count;         /* [R,R] tokens of source rank s received by rank r,
                                             or NULL; needs R | T                        */
    int32_t* token_offset;          /* [T+1] exclusive prefix over tokens of n(t) (rows
                                             numbered token by token; [T] = N), or NULL.
                                             The bulk-copy dispatch alternative uses it
                                             to give every CTA the same number of rows  */
    int32_t* expanded_row;          /* [T,K] expanded (per-expert) row of each valid
                                             (t, k), -1 if masked, or NULL; see
                                             ep_dispatch_expanded                        */
    int32_t* node_offset;           /* [nodes+1] exclusive prefix of num_tokens_per_node
                                             (nodes = R / ranks_per_node), or NULL       */
    int32_t* node_row;              /* [T,nodes] row of token t in node n's scale-out
                                             buffer or -1; rows of node n are
                                             node_offset[n] + 0, 1, ... in ascending t.
                                             NULL, or set together with node_offset and
                                             num_tokens_per_node (ranks_per_node > 0;
                                             with no tokens node_row may be NULL and
                                             node_offset is all zero);
                                             see ep_dispatch_hierarchical              */
} ep_layout_t;

/* Bytes of device workspace ep_get_layout needs for these sizes (>= 16). */
size_t ep_layout_workspace_bytes(int num_tokens, int num_topk, int num_experts, int num_ranks,
                                 int ranks_per_node);

/* An upper bound on N: num_tokens * min(num_topk, num_ranks).  A receive
 * buffer of this many rows never overflows ("DeepEP V2 ElasticBuffer
 * architecture", calculate_buffer_size fragment: size buffers for the worst
 * case so that no host wait is needed before dispatch). */
int64_t ep_recv_capacity_bound(int num_tokens, int num_topk, int num_ranks);

/*
 * Routing layout ("DeepEP Symmetric Memory" sections 6.1 and 7.3).
 *
 * topk_idx        int64 [T,K]: expert of each top-k slot, -1 = masked.  Entries
 *                 outside [-1, E) set EP_ERR_INVALID_INDEX and are skipped.
 *                 A repeated expert counts once per entry in
 *                 num_tokens_per_expert and once for its rank.
 * ranks_per_node  0 = no node counts; else must divide R, and when
 *                 out->num_tokens_per_node is non-NULL it receives, per group of
 *                 ranks_per_node consecutive ranks, the tokens with any expert
 *                 in that group.
 * expert_alignment >= 1; only expert_offset uses it.
 * out             the layout arrays (num_tokens_per_node, src_dst_count,
 *                 token_offset and expanded_row may be NULL; src_dst_count
 *                 non-NULL needs R | T).  expanded_row: expert e's valid
 *                 (t, k) entries take rows expert_offset[e] + 0, 1, ... in
 *                 (token, k) order; rows between expert e's count and the next
 *                 aligned offset are padding.
 * workspace       device scratch of ws_bytes >= ep_layout_workspace_bytes(...);
 *                 its contents need no initialisation and are garbage after.
 * Results depend only on topk_idx (no atomics decide any order).
 */
ep_status_t ep_get_layout(const int64_t* topk_idx, int num_tokens, int num_topk, int num_experts,
                          int num_ranks, int ranks_per_node, int expert_alignment,
                          const ep_layout_t* out, void* workspace, size_t ws_bytes,
                          int32_t* d_status, void* cuda_stream);

/* Size of the library's built-in layout scratch (4 MiB). */
#define EP_LAYOUT_STATIC_SCRATCH_BYTES (4u << 20)

/*
 * Routing layout without a caller workspace.  The pages have no counterpart:
 * this is a library convenience.
 *
 * For callers that cannot allocate device memory: a plugin that a host
 * framework hands only its input and output buffers, with no allocator of its
 * own, or a process whose device memory is fully reserved up front by a
 * pooling allocator, so that a further cudaMalloc fails or is not allowed.
 * Same arguments and results as ep_get_layout minus `workspace` / `ws_bytes`:
 * the scratch is a device array of EP_LAYOUT_STATIC_SCRATCH_BYTES built into
 * the library, which every GPU that loads the library holds until the process
 * exits.  The call allocates nothing.
 *
 * Arguments are checked exactly as by ep_get_layout (same codes); then, before
 * any launch, the call returns EP_ERR_UNSUPPORTED when
 * ep_layout_workspace_bytes(num_tokens, num_topk, num_experts, num_ranks,
 * ranks_per_node) > EP_LAYOUT_STATIC_SCRATCH_BYTES (for example T=32768,
 * E=256, R=64 needs about 0.43 MB; T=16384, E=2048, R=1024 about 2.9 MB).
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress, which allocates nothing) and returns EP_ERR_CUDA if
 * that fails; the first call on a device also loads the library's device
 * code there, so make it before any stream capture.  All calls share the one
 * array, and every call overwrites the scratch words it reads, so nothing
 * needs clearing between calls; but calls whose kernels overlap on the GPU
 * (on unordered streams) race on it and give wrong layouts: order them.
 */
ep_status_t ep_get_layout_static_scratch(const int64_t* topk_idx, int num_tokens, int num_topk,
                                         int num_experts, int num_ranks, int ranks_per_node,
                                         int expert_alignment, const ep_layout_t* out,
                                         int32_t* d_status, void* cuda_stream);

/*
 * Dispatch ("DeepEP Symmetric Memory" sections 6.1 and 9.2; "DeepEP V2
 * ElasticBuffer architecture", TokenLayout fragment).  For every token t and
 * rank r with dst_row[t,r] = d >= 0:
 *   recv_x[d]               = x[t] (bf16 copy), or its FP8 E4M3 cast;
 *   recv_sf[d, b]           = FP8 scale of 128-channel block b (FP8 only);
 *   recv_topk_idx[d, k]     = topk_idx[t,k] - r*E_l if that expert is on r, else -1;
 *   recv_topk_weights[d, k] = topk_weights[t,k] if that expert is on r, else 0;
 *   recv_src_idx[d]         = t.
 * FP8 cast per token and 128-channel block: amax = max |x|; scale
 * sf = amax/448 and codes e4m3_rne_satfinite(x * (448/amax)), both fp32 IEEE;
 * an all-zero block has sf = 1 and codes of +-0.
 *
 * x                 [T,H] bf16 (any 2-byte payload is copied bit for bit).
 * topk_idx          int64 [T,K]; topk_weights fp32 [T,K] (may be NULL when
 *                   recv_topk_weights is NULL).
 * layout            from ep_get_layout for the same topk_idx (only dst_row is read).
 * out_dtype         EP_BF16 (H % 8 == 0) or EP_FP8_E4M3 (H % 128 == 0).
 * recv_capacity     rows allocated in every recv_* array; a row d >= capacity
 *                   is skipped and sets EP_ERR_CAPACITY.
 * recv_x            [capacity, H] of 2-byte (bf16) or 1-byte (FP8) elements.
 * recv_sf           FP8 only: fp32 scales, row-major [capacity, H/128] when
 *                   sf_col_major == 0, else element (d, b) at b*sf_stride + d
 *                   with sf_stride = capacity rounded up to a multiple of 4
 *                   (a column-major layout a following GEMM can load by TMA).
 * recv_topk_idx     int32 [capacity, K] or NULL; recv_topk_weights fp32
 *                   [capacity, K] or NULL; recv_src_idx int32 [capacity] or NULL.
 * num_sms           0 = use the whole GPU; n > 0 = SM-limited mode: a
 *                   persistent grid of min(n, SMs) CTAs, one per SM, so the
 *                   copy can overlap compute kernels on the other SMs ("DeepEP V2
 *                   ElasticBuffer architecture", get_theoretical_num_sms: the
 *                   SM count is chosen to leave the rest to compute).  Results
 *                   are identical in both modes.  The same argument exists on
 *                   ep_combine, ep_dispatch_expanded and ep_combine_expanded.
 */
ep_status_t ep_dispatch(const void* x, const int64_t* topk_idx, const float* topk_weights,
                        int num_tokens, int hidden, int num_topk, int num_experts, int num_ranks,
                        const ep_layout_t* layout, int out_dtype, int64_t recv_capacity,
                        void* recv_x, float* recv_sf, int sf_col_major,
                        int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* recv_src_idx,
                        int num_sms, int32_t* d_status, void* cuda_stream);

/*
 * Layout and dispatch in one call: the pages' dispatch, which computes the
 * routing handle itself ("DeepEP Symmetric Memory" section 9.2,
 * dispatch(x, topk_idx, topk_weights, num_experts, ...) -> (recv_x, ...,
 * handle); section 6.1 for the prefix sums it launches with).
 *
 * Same results as ep_get_layout followed by ep_dispatch with num_sms = 0:
 * `layout` receives every array ep_get_layout writes, and the receive arrays
 * what ep_dispatch writes.  Arguments are those two calls' arguments
 * (num_tokens .. num_ranks, ranks_per_node and expert_alignment as in
 * ep_get_layout; out_dtype .. recv_src_idx as in ep_dispatch), checked on the
 * host before anything is launched.  Since N is not known before the
 * layout, size the receive arrays with ep_recv_capacity_bound.
 *
 * With few tokens (1 <= num_tokens <= 256, num_ranks <= 32, num_topk <= 16,
 * num_experts <= 2048, and no expanded or node rows requested in `layout`)
 * the call launches a single kernel: each dispatch CTA derives its token's
 * destination rows from topk_idx by the layout's definition (rank offset plus
 * the number of earlier tokens on that rank) and writes the token's layout
 * rows, and two more CTAs write the layout's counts and offsets, so no
 * layout kernel runs in front of the dispatch (the workspace is then not
 * touched).  This shortens the latency-bound decode step.  Otherwise the call
 * launches the layout kernel(s) and then the dispatch, as the two separate
 * calls do.  Where the layout is the one-cluster kernel (up to 2^19 token-rank
 * pairs beyond the few-token case) and the workspace is 128-byte aligned
 * with room for one 128-byte line per cluster CTA (at most 2 KiB), each layout
 * CTA also publishes in its line when its block of dst_row is written, and
 * the dispatch CTAs of the first wave start on that instead of on the layout
 * kernel's completion; the dispatch's last CTA clears the lines, so a CUDA
 * graph may replay the call.  The workspace then belongs to the call until
 * the dispatch completes, and its contents are garbage after, as for
 * ep_get_layout.
 */
ep_status_t ep_layout_and_dispatch(const void* x, const int64_t* topk_idx, const float* topk_weights,
                                   int num_tokens, int hidden, int num_topk, int num_experts,
                                   int num_ranks, int ranks_per_node, int expert_alignment,
                                   const ep_layout_t* layout, void* workspace, size_t ws_bytes,
                                   int out_dtype, int64_t recv_capacity, void* recv_x, float* recv_sf,
                                   int sf_col_major, int32_t* recv_topk_idx, float* recv_topk_weights,
                                   int32_t* recv_src_idx, int32_t* d_status, void* cuda_stream);

/*
 * Combine ("DeepEP Symmetric Memory" section 9.2: combine(x, handle,
 * topk_weights) -> combined_x).  For every token t:
 *   out[t] = bf16_rne( sum over r with dst_row[t,r] = d >= 0 of c(t,r) * y[d] )
 * accumulated in fp32, with c = 1 when topk_weights is NULL (unweighted), else
 * c(t,r) = sum of topk_weights[t,k] over the k whose expert is on r.  A token
 * in no rank gets a zero row.
 *
 * y           bf16 [num_y_rows, H]: the expert outputs, in the receive rows of
 *             dispatch; a row d >= num_y_rows is skipped (EP_ERR_CAPACITY).
 * topk_idx    int64 [T,K]; needed when topk_weights is non-NULL.
 * out         bf16 [T,H].  H % 8 == 0.
 */
ep_status_t ep_combine(const void* y, int64_t num_y_rows, const int64_t* topk_idx,
                       const float* topk_weights, int num_tokens, int hidden, int num_topk,
                       int num_experts, int num_ranks, const ep_layout_t* layout, void* out,
                       int num_sms, int32_t* d_status, void* cuda_stream);

/*
 * Expanded (per-expert) receive layout ("DeepEP V2 ElasticBuffer
 * architecture": the dispatch_copy_epilogue and combine_reduce_epilogue
 * kernels and the TokenLayout record's linked_list_idx; "DeepEP Symmetric
 * Memory" section 6.1: expert_alignment and the unaligned per-expert counts).
 * Every valid top-k slot (t, k) gets its own row, grouped by expert (the
 * experts of rank 0, then rank 1, ...) and padded so that expert e's block
 * starts at expert_offset[e] -- the input of a grouped GEMM.  In one GPU's
 * memory the pages' two steps (rank rows, then a per-expert copy epilogue;
 * a per-expert weighted reduce, then the rank return) are done directly.
 *
 * Bound on the rows: T*K + E*(expert_alignment - 1); the exact count is
 * expert_offset[E].
 */
int64_t ep_expanded_capacity_bound(int num_tokens, int num_topk, int num_experts,
                                   int expert_alignment);

/*
 * Expanded dispatch: for every (t, k) with d = layout->expanded_row[t,k] >= 0:
 *   recv_x[d] = x[t] (bf16 copy) or its FP8 E4M3 cast (same cast as
 *   ep_dispatch; recv_sf row-major or column-major as there);
 *   recv_src_idx[d] = t; recv_weight[d] = topk_weights[t,k].
 * Padding rows are not written.  layout must come from ep_get_layout with
 * expanded_row set.  recv_src_idx / recv_weight may be NULL (recv_weight
 * non-NULL needs topk_weights).  Other arguments and errors as ep_dispatch.
 */
ep_status_t ep_dispatch_expanded(const void* x, const int64_t* topk_idx, const float* topk_weights,
                                 int num_tokens, int hidden, int num_topk, int num_experts,
                                 int num_ranks, const ep_layout_t* layout, int out_dtype,
                                 int64_t recv_capacity, void* recv_x, float* recv_sf, int sf_col_major,
                                 int32_t* recv_src_idx, float* recv_weight, int num_sms,
                                 int32_t* d_status, void* cuda_stream);

/*
 * Expanded combine: out[t] = bf16_rne( sum over k ascending with
 * d = layout->expanded_row[t,k] >= 0 of c * y[d] ), fp32 accumulation,
 * c = topk_weights[t,k], or 1 when topk_weights is NULL.  The per-(token,
 * slot) weighting and the reduction over slots and ranks in one pass.
 * y bf16 [num_y_rows, H]; rows >= num_y_rows are skipped (EP_ERR_CAPACITY).
 */
ep_status_t ep_combine_expanded(const void* y, int64_t num_y_rows, const float* topk_weights,
                                int num_tokens, int hidden, int num_topk, int num_experts,
                                int num_ranks, const ep_layout_t* layout, void* out, int num_sms,
                                int32_t* d_status, void* cuda_stream);

/*
 * Combined top-k weights ("DeepEP Symmetric Memory" section 9.2: combine
 * returns combined_topk_weights).  For every token t and slot k:
 *   combined_topk_weights[t,k] = sum over ranks r holding t (ascending, fp32)
 *                                of recv_topk_weights[dst_row[t,r], k].
 * Each slot's weight travels only in the row of the rank holding its expert,
 * so for received weights that were not modified this returns topk_weights for
 * valid slots and 0 for masked ones.  recv_topk_weights fp32 [num_rows, K]
 * (as written by ep_dispatch, possibly updated by the experts);
 * combined_topk_weights fp32 [T, K].  Rows >= num_rows set EP_ERR_CAPACITY.
 */
ep_status_t ep_combine_topk_weights(const float* recv_topk_weights, int64_t num_rows, int num_tokens,
                                    int num_topk, int num_experts, int num_ranks,
                                    const ep_layout_t* layout, float* combined_topk_weights,
                                    int32_t* d_status, void* cuda_stream);

/*
 * Cumulative receive statistics ("DeepEP Symmetric Memory" section 6.1:
 * cumulative_local_expert_recv_stats, a load-balance monitor): adds the
 * layout's num_tokens_per_expert to the caller's int64 counters stats[E].
 */
ep_status_t ep_accumulate_expert_stats(const ep_layout_t* layout, int num_experts, int64_t* stats,
                                       void* cuda_stream);

/*
 * Hierarchical (two-stage) dispatch ("DeepEP V2 ElasticBuffer architecture":
 * hybrid_dispatch, the path taken when there is more than one scale-out
 * domain; the WorkspaceLayout fragment keeps scale-out rank counts beside the
 * scale-up ones; node = rank / ranks_per_node as in "V1 Buffer
 * initialisation" section 3.2).  Node n holds ranks [n*rpn, (n+1)*rpn).
 *
 * Stage 1 (scale-out): each token goes once to every node holding one of its
 * experts:  node_x[j] = x[t] (bf16) or its FP8 cast (codes, with row-major
 * scales node_sf[j, H/128]), node_src_idx[j] = t, for j = node_row[t,n] >= 0.
 * Stage 2 (scale-up): each node row is copied to the ranks r of its node with
 * dst_row[t,r] >= 0, with the per-row metadata of ep_dispatch.  recv_* end up
 * identical to ep_dispatch's (same arguments, layout and capacity).
 *
 * layout          from ep_get_layout with node_row / node_offset set (same
 *                 ranks_per_node).
 * node_capacity   rows of node_x / node_sf / node_src_idx; node_offset[nodes]
 *                 rows are used, at most T * min(K, nodes)
 *                 (= ep_recv_capacity_bound(T, K, nodes)).  Rows at or beyond
 *                 it set EP_ERR_CAPACITY and are skipped.
 * node_x          bf16 [node_capacity, H] or FP8 codes [node_capacity, H];
 *                 node_sf fp32 [node_capacity, H/128] (FP8, required);
 *                 node_src_idx int32 [node_capacity] or NULL.
 * Other arguments and errors as ep_dispatch (no SM-limited mode).  Two kernel
 * launches on the stream; the node buffers are the caller's.
 */
ep_status_t ep_dispatch_hierarchical(const void* x, const int64_t* topk_idx, const float* topk_weights,
                                     int num_tokens, int hidden, int num_topk, int num_experts,
                                     int num_ranks, int ranks_per_node, const ep_layout_t* layout,
                                     int out_dtype, int64_t node_capacity, void* node_x, float* node_sf,
                                     int32_t* node_src_idx, int64_t recv_capacity, void* recv_x,
                                     float* recv_sf, int sf_col_major, int32_t* recv_topk_idx,
                                     float* recv_topk_weights, int32_t* recv_src_idx, int32_t* d_status,
                                     void* cuda_stream);

/*
 * Hierarchical (two-stage) combine ("DeepEP V2 ElasticBuffer architecture":
 * hybrid_combine), the reverse of ep_dispatch_hierarchical.
 * Stage 1 (scale-up reduce): for every (t, n) with j = node_row[t,n] >= 0,
 *   node_y[j] = bf16( sum over ranks r of node n holding t of c(t,r) *
 *   y[dst_row[t,r]] ), fp32 accumulation, c as in ep_combine.
 * Stage 2 (scale-out reduce): out[t] = bf16( sum over nodes of node_y[j] ),
 *   fp32 accumulation.
 * The node partial is rounded to bf16 (the data type on the scale-out link),
 * so the result may differ from ep_combine by the rounding of each partial.
 * y bf16 [num_y_rows, H]; node_y bf16 [node_capacity, H] (the caller's
 * buffer); out bf16 [T, H].  Rows beyond num_y_rows or node_capacity set
 * EP_ERR_CAPACITY and are skipped.  Other arguments as ep_combine.
 */
ep_status_t ep_combine_hierarchical(const void* y, int64_t num_y_rows, const int64_t* topk_idx,
                                    const float* topk_weights, int num_tokens, int hidden, int num_topk,
                                    int num_experts, int num_ranks, int ranks_per_node,
                                    const ep_layout_t* layout, int64_t node_capacity, void* node_y, void* out,
                                    int32_t* d_status, void* cuda_stream);

/*
 * SM count rule for the SM-limited mode ("DeepEP V2 ElasticBuffer
 * architecture", get_theoretical_num_sms and its get_expected_topk helper),
 * restated for ranks that share one HBM.  Host-only arithmetic, no GPU call.
 *
 *   g     = R * (1 - C(E - E/R, K) / C(E, K))   expected ranks per token when
 *           each token picks K distinct experts uniformly at random
 *   bytes the SMs move per token (payload only):
 *           dispatch: read 2H, write g * row, row = 2H (bf16) or
 *                     H + 4*H/128 (FP8 codes + fp32 scales)
 *           combine:  read g * 2H, write 2H
 *   the bounding link is the HBM itself (hbm_gbs), carrying read + write, so
 *   n     = max(hbm_gbs / (read + write) * read  / sm_read_gbs,
 *               hbm_gbs / (read + write) * write / sm_write_gbs)
 *   n     = max(4, ceil(1.25 * n)) rounded up to even; at least 64 when
 *           prefer_overlap_with_compute == 0; at most device_sms.
 *
 * The pages' per-SM rates are sm_read_gbs = 200 and sm_write_gbs = 50.
 * is_combine: 0 = dispatch, 1 = combine (combine reads bf16 rows whatever
 * out_dtype is).  Returns the SM count, or 0 for invalid arguments (hidden not
 * a positive multiple of 128 for FP8 or of 8 otherwise, K outside 1..min(E, 32),
 * R not dividing E, a rate or device_sms not positive).
 */
int ep_theoretical_num_sms(int hidden, int num_topk, int num_experts, int num_ranks, int out_dtype,
                           int is_combine, double hbm_gbs, double sm_read_gbs, double sm_write_gbs,
                           int prefer_overlap_with_compute, int device_sms);

/* Text for a status word (bits joined by '|'); a static string. */
const char* ep_status_string(int32_t status);

/* ABI version of this header (bumped on any signature change). */
int ep_abi_version(void);

/* 1 when this copy of the library is the bounds-checked build (every kernel
 * compiled with EP_GET_CHECKED=1: each global load and store is checked
 * against the extent its arguments declare, a failing access is skipped and
 * sets EP_ERR_OUT_OF_BOUNDS in *d_status), 0 for the product build.  The
 * checked build computes the same results on valid input, more slowly. */
int ep_bounds_checked(void);

#ifdef __cplusplus
}
#endif

#endif /* EP_GET_H */
