// Internal declarations shared by the CUDA translation units of libep_get.so:
// kernel parameter blocks, launchers, and thin inline-PTX wrappers for the
// Blackwell bulk-copy engine (cp.async.bulk + mbarrier) and streaming loads.
#pragma once

#include <cstdint>
#include <cstddef>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/ep_get.h"

namespace epg {

// ---------------------------------------------------------------------------
// Parameter blocks
// ---------------------------------------------------------------------------

constexpr int kTileTokens = 256;               // tokens per layout tile (one per thread)
// ep_layout_and_dispatch: one kernel computes layout and dispatch (each CTA
// derives its token's rows itself) for at most this many tokens, top-k
// entries per token and experts, with R <= 32
constexpr int kSelfRouteMaxTokens = 256;
constexpr int kSelfRouteMaxTopk = 16;
constexpr int kSelfRouteMaxExperts = 2048;
constexpr int kTileWords = kTileTokens / 32;   // 32-bit membership words per rank per tile

// Rows-ready signal of ep_layout_and_dispatch on the cluster layout path, in
// the caller's workspace (which that path does not otherwise use): one
// 128-byte line per layout CTA.  Word 0 holds the call's tag once the CTA's
// block of dst_row is written; the low 32 bits of word 1 count the dispatch
// CTAs that have looked for it.  The layout CTA clears the count before it
// publishes the tag; the dispatch grid's last CTA, once the layout kernel has
// completed and every reader has counted itself, clears the tag, so a line
// holds no tag between calls (a CUDA graph replays a call with the same
// tag).  A dispatch CTA that sees no tag within kRowsWaitNs waits for the
// layout kernel's completion instead.
constexpr int kReadyWords = 16;   // 64-bit words per slot line
#ifndef EP_ROWS_WAIT_NS
#define EP_ROWS_WAIT_NS 200000ull
#endif
constexpr uint64_t kRowsWaitNs = EP_ROWS_WAIT_NS;
struct RowsSignal {
    uint64_t* slots;   // in: the workspace, or null for no signal; out: null when the layout does not publish
    uint64_t tag;      // in: this call's tag (never 0)
    size_t bytes;      // in: workspace bytes available for slot lines
    int tokens;        // out: tokens per slot (one layout CTA's range)
    int count;         // out: slots
};

struct LayoutParams {
    const int64_t* topk_idx;
    int T, K, E, R, experts_per_rank, ranks_per_node, num_nodes, alignment, num_tiles;
    int32_t* num_tokens_per_rank;
    int32_t* num_tokens_per_node;
    int32_t* num_tokens_per_expert;
    uint8_t* is_token_in_rank;
    int32_t* rank_offset;
    int32_t* expert_offset;
    int32_t* dst_row;
    int32_t* src_dst_count;
    int32_t* token_offset;
    int32_t* expanded_row;   // [T][K] or null
    int32_t* node_offset;    // [num_nodes + 1] or null (set together with node_row)
    int32_t* node_row;       // [T][num_nodes] or null
    // workspace
    int32_t* ws_rank;      // [R][num_tiles]: tile counts, then exclusive tile prefix
    int32_t* ws_expert;    // [E][num_tiles]
    int32_t* ws_node;      // [num_nodes][num_tiles]
    uint32_t* ws_bitmap;   // [num_tiles][kTileWords][R]
    int32_t* status;
    uint64_t* rows_ready;  // cluster path: publish each CTA's rows here (null: no signal)
    uint64_t rows_tag;
};

struct DispatchParams {
    const uint8_t* x;
    const int64_t* topk_idx;
    const float* topk_weights;
    const int32_t* dst_row;
    const int32_t* token_offset;   // may be null
    const int32_t* expanded_row;   // expanded mode: [T][K] destination rows instead of dst_row
    float* recv_weight;            // expanded mode: weight of each received (token, k)
    int T, H, K, E, R, experts_per_rank;
    int64_t capacity;
    uint8_t* recv_x;
    float* recv_sf;
    int sf_col_major;
    int64_t sf_stride;
    int32_t* recv_topk_idx;
    float* recv_topk_weights;
    int32_t* recv_src_idx;
    int32_t* status;
    int num_sms;            // > 0: SM-limited mode (persistent CTAs, one per SM)
    // work split: each token row is cut into `chunks` pieces
    int chunks;
    uint32_t chunk_bytes;   // bf16 path: bytes per piece (multiple of 16)
    int chunk_blocks;       // fp8 path: 128-channel blocks per piece
    // L2 prefetch of x before the wait on the previous kernel: CTA b <
    // prefetch_ctas prefetches the pieces of items b + j * prefetch_ctas,
    // j < prefetch_items (0: none)
    int prefetch_ctas;
    int prefetch_items;
    int prefetch_evict_last;   // 1: the prefetch is evict-last, only the first wave prefetches, and a
                               // read piece of x goes back to the normal priority
    // 1: ep_layout_and_dispatch with few tokens: no layout kernel runs; each
    // CTA derives its token's destination rows from topk_idx, writes that
    // token's layout rows, and two extra CTAs the layout's counts and
    // offsets, into:
    int self_route;
    int32_t* l_num_tokens_per_rank;     // [R]
    int32_t* l_num_tokens_per_node;     // [R / ranks_per_node] or null
    int32_t* l_num_tokens_per_expert;   // [E]
    uint8_t* l_is_token_in_rank;        // [T][R]
    int32_t* l_rank_offset;             // [R + 1]
    int32_t* l_expert_offset;           // [E + 1]
    int32_t* l_dst_row;                 // [T][R]
    int32_t* l_src_dst_count;           // [R][R] or null
    int32_t* l_token_offset;            // [T + 1] or null
    int l_alignment, l_ranks_per_node, l_num_nodes;
    // rows-ready signal (one item per CTA, rank rows): the CTAs below
    // rows_first_wave (the first wave, which starts while the layout kernel
    // runs) wait for the tag in slot t / rows_tokens instead of the layout
    // kernel's completion
    uint64_t* rows_ready;
    uint64_t rows_tag;
    int rows_tokens, rows_slots, rows_first_wave;
};

struct CombineParams {
    const uint8_t* y;
    int64_t num_y_rows;
    const int64_t* topk_idx;
    const float* topk_weights;
    const int32_t* dst_row;
    const int32_t* expanded_row;   // expanded mode: [T][K] source rows instead of dst_row
    int T, H, K, E, R, experts_per_rank;
    uint8_t* out;
    int32_t* status;
    int chunks;             // pieces per token row
    int chunk_vecs;         // 16-byte vectors per piece
    int num_sms;            // > 0: SM-limited mode (persistent CTAs, one per SM)
};

// Hierarchical path, the scale-up halves (the scale-out halves reuse the
// dispatch and combine kernels with node_row in place of dst_row).
struct HierParams {
    const uint8_t* node_x;        // forward: node rows, row_bytes each
    const float* node_sf;         // forward, FP8: [node_capacity][H/128]
    const int64_t* topk_idx;
    const float* topk_weights;
    const int32_t* dst_row;       // [T][R]
    const int32_t* node_row;      // [T][num_nodes]
    int T, H, K, E, R, experts_per_rank, ranks_per_node, num_nodes;
    int64_t node_capacity;
    // forward (dispatch stage 2)
    int64_t capacity;
    uint8_t* recv_x;
    float* recv_sf;
    int sf_col_major;
    int64_t sf_stride;
    int32_t* recv_topk_idx;
    float* recv_topk_weights;
    int32_t* recv_src_idx;
    // reduce (combine stage 1)
    const uint8_t* y;
    int64_t num_y_rows;
    uint8_t* node_y;
    int32_t* status;
    int chunks;             // pieces per row
    uint32_t chunk_bytes;   // forward: bytes per piece (multiple of 16)
    int chunk_vecs;         // reduce: 16-byte vectors per piece
};

struct CombineWeightsParams {
    const float* recv_topk_weights;
    int64_t num_rows;
    const int32_t* dst_row;
    int T, K, R;
    float* combined;
    int32_t* status;
};

struct DeviceInfo {
    int device;
    int num_sms;
    int max_smem_optin;
};

// Cached per-device properties (host).
const DeviceInfo& device_info();

// Launchers (host).  Each returns cudaSuccess or the launch error.
// sig (ep_layout_and_dispatch): on the cluster path with room for its slot
// lines the layout CTAs publish their rows; otherwise sig->slots is cleared.
cudaError_t launch_layout(const LayoutParams& p, cudaStream_t stream, RowsSignal* sig = nullptr);
cudaError_t launch_dispatch_bf16(DispatchParams p, cudaStream_t stream);
cudaError_t launch_dispatch_fp8(DispatchParams p, cudaStream_t stream);
// True when the dispatch that ep_layout_and_dispatch launches on the layout
// kernel's rows (num_sms 0, not self-routed) waits for the rows-ready signal.
bool dispatch_reads_rows_signal(bool fp8);
cudaError_t launch_combine(CombineParams p, bool weighted, cudaStream_t stream);
cudaError_t launch_combine_topk_weights(const CombineWeightsParams& p, cudaStream_t stream);
cudaError_t launch_accumulate_expert_stats(const int32_t* counts, int E, int64_t* stats, cudaStream_t stream);
cudaError_t launch_forward_scaleup(HierParams p, bool fp8, cudaStream_t stream);
cudaError_t launch_reduce_scaleup(HierParams p, bool weighted, cudaStream_t stream);

// Host-side logging, on when EP_GET_DEBUG is set to anything but "0" (read
// once per process): one line on stderr per C-ABI call, per argument check
// that rejects a call (with the check's line in api.cu) and per kernel launch
// (kernel, grid, block, dynamic shared memory, cluster size).
bool debug_enabled();
void debug_log(const char* fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 1, 2)))
#endif
    ;
void debug_launch(const void* kernel, dim3 grid, dim3 block, size_t smem, int cluster);
#define EP_DEBUG(...)                                                 \
    do {                                                              \
        if (::epg::debug_enabled()) ::epg::debug_log(__VA_ARGS__);   \
    } while (0)

// Launch with programmatic dependent launch allowed: the kernel may begin
// while the previous kernel on the stream is still running, and must call
// pdl_wait() before it reads anything that kernel writes.  After any other
// stream operation the attribute has no effect.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (debug_enabled()) debug_launch(reinterpret_cast<const void*>(kernel), grid, block, smem, 1);
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Host checks of ep_get_layout (every argument; the workspace too when
// check_workspace) and its parameter block, without a launch.
ep_status_t layout_params(const int64_t* topk_idx, int T, int K, int E, int R, int ranks_per_node,
                          int expert_alignment, const ep_layout_t* out, void* workspace, size_t ws_bytes,
                          int32_t* d_status, bool check_workspace, LayoutParams& p);

// Workspace carve-up shared by the size query and the launcher.
struct LayoutWorkspace {
    size_t off_rank, off_expert, off_node, off_bitmap, total;
};
LayoutWorkspace layout_workspace(int T, int E, int R, int num_nodes);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Bounds-checked build (compiled with -DEP_GET_CHECKED=1; a test-only copy of
// the library, never the product): in_bounds(i, n, status) is true when
// 0 <= i < n; otherwise it ORs EP_ERR_OUT_OF_BOUNDS into *status and is
// false, and the caller skips the access.  The product build compiles it to
// the constant true, so its code is unchanged.
#ifndef EP_GET_CHECKED
#define EP_GET_CHECKED 0
#endif
__device__ __forceinline__ bool in_bounds(int64_t i, int64_t n, int32_t* status) {
#if EP_GET_CHECKED
    if (i >= 0 && i < n) return true;
    atomicOr(status, EP_ERR_OUT_OF_BOUNDS);
    return false;
#else
    (void)i;
    (void)n;
    (void)status;
    return true;
#endif
}
// Element i of an array of n, and a byte range [off, off + len) of an
// array of n bytes, against the kernel's parameter block `p` (its status).
#define EP_IN(i, n) ::epg::in_bounds(static_cast<int64_t>(i), static_cast<int64_t>(n), p.status)
#define EP_IN_BYTES(off, len, n) \
    ::epg::in_bounds(static_cast<int64_t>(off), static_cast<int64_t>(n) - static_cast<int64_t>(len) + 1, p.status)
// A row index read from dst_row / expanded_row / node_row: -1 (absent) or >= 0.
#define EP_ROW_OK(d) ((d) >= -1 || ::epg::in_bounds(-1, 0, p.status))

// A bounded wait gives up after this many nanoseconds of %globaltimer (the
// failure-path test builds a copy of the library with a shorter limit).
#ifndef EP_WAIT_TIMEOUT_NS
#define EP_WAIT_TIMEOUT_NS 2000000000ull
#endif
constexpr uint64_t kWaitTimeoutNs = EP_WAIT_TIMEOUT_NS;

// Wait until the kernel this one depends on (previous on the stream) has
// completed and its writes are visible; returns at once without a dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel on the stream to be scheduled now (it still waits in
// pdl_wait() for this kernel to complete before reading its outputs).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false after the
// timeout (the caller records EP_ERR_TIMEOUT and winds down).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < (1u << 30); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0 && global_timer_ns() - t0 > kWaitTimeoutNs) return false;
    }
    return false;
}

// Bulk copy global -> shared; completion is signalled on `bar` as tx bytes.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Bulk copy shared -> global, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}

// L2 policy that marks lines for early eviction.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy that keeps lines ahead of normal and evict-first ones.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Back to the normal eviction priority for the 128-byte L2 line at p.
__device__ __forceinline__ void l2_priority_normal(const void* p) {
    asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(p) : "memory");
}

// 16-byte store with an L2 cache policy.
__device__ __forceinline__ void st_v4_hint(void* p, uint4 v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}

// Bulk copy shared -> global with an L2 cache policy.
__device__ __forceinline__ void bulk_store_evict_first(void* dst, const void* src_smem, uint32_t bytes,
                                                       uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(smem_addr(src_smem)), "r"(bytes), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk groups are still reading smem.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are still in flight.
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Loads, stores and counts of the rows-ready signal (memory-model strong, at
// GPU scope).
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_relaxed_add_u32(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16-byte read-only streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Barrier over `threads` threads of the CTA on hardware barrier `id` (1..15;
// 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 16-byte streaming store (evict-first at every cache level).
__device__ __forceinline__ void st_cs_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ int warp_inclusive_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

}  // namespace epg
