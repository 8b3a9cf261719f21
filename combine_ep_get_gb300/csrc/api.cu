// C ABI of libep_get.so: host-side argument checks, parameter blocks and
// launches.  Declarations and the full contract are in include/ep_get.h.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cxxabi.h>
#include <mutex>
#include <string>

#include "ep_internal.cuh"

namespace epg {

bool debug_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("EP_GET_DEBUG");
        return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
    }();
    return on;
}

void debug_log(const char* fmt, ...) {
    char line[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(line, sizeof(line), fmt, ap);
    va_end(ap);
    std::fprintf(stderr, "[ep_get] %s\n", line);
}

void debug_launch(const void* kernel, dim3 grid, dim3 block, size_t smem, int cluster) {
    const char* name = nullptr;
    if (cudaFuncGetName(&name, kernel) != cudaSuccess || name == nullptr) {
        cudaGetLastError();
        name = "?";
    }
    int st = 0;
    char* readable = abi::__cxa_demangle(name, nullptr, nullptr, &st);
    debug_log("launch %s grid (%u, %u, %u) block (%u, %u, %u) smem %zu cluster %d",
              (st == 0 && readable) ? readable : name, grid.x, grid.y, grid.z, block.x, block.y, block.z, smem,
              cluster);
    std::free(readable);
}

// A status a host check returns, logged (with the check's line) when it is an error.
ep_status_t debug_ret(const char* fn, int line, ep_status_t s) {
    if (s != EP_OK && debug_enabled()) debug_log("%s: %s (api.cu:%d)", fn, ep_status_string(s), line);
    return s;
}

const DeviceInfo& device_info() {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static DeviceInfo infos[kMaxDevices];
    static bool have[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d{dev, 0, 0};
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (d.num_sms < 1) d.num_sms = 1;
        infos[dev] = d;
        have[dev] = true;
    }
    return infos[dev];
}

}  // namespace epg

#define EP_RET(s) ::epg::debug_ret(__func__, __LINE__, (s))

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

// Shape checks shared by the three calls.
ep_status_t check_shape(int T, int K, int E, int R) {
    if (T < 0 || K < 1 || E < 1 || R < 1) return EP_RET(EP_ERR_INVALID_ARG);
    if (K > EP_MAX_TOPK || R > EP_MAX_RANKS || E > EP_MAX_EXPERTS) return EP_RET(EP_ERR_UNSUPPORTED);
    if (E % R != 0) return EP_RET(EP_ERR_INVALID_ARG);
    if (E / R > EP_MAX_EXPERTS_PER_RANK) return EP_RET(EP_ERR_UNSUPPORTED);
    if (static_cast<int64_t>(T) * R > INT32_MAX || static_cast<int64_t>(T) * K > INT32_MAX)
        return EP_RET(EP_ERR_UNSUPPORTED);
    return EP_OK;
}

}  // namespace

extern "C" {

int ep_abi_version(void) { return 8; }

int ep_bounds_checked(void) { return EP_GET_CHECKED ? 1 : 0; }

size_t ep_layout_workspace_bytes(int num_tokens, int num_topk, int num_experts, int num_ranks,
                                 int ranks_per_node) {
    (void)num_topk;
    if (num_tokens < 0 || num_experts < 1 || num_ranks < 1) return 16;
    const int nodes = ranks_per_node > 0 ? num_ranks / ranks_per_node : 0;
    return epg::layout_workspace(num_tokens, num_experts, num_ranks, nodes).total;
}

int ep_theoretical_num_sms(int hidden, int num_topk, int num_experts, int num_ranks, int out_dtype,
                           int is_combine, double hbm_gbs, double sm_read_gbs, double sm_write_gbs,
                           int prefer_overlap_with_compute, int device_sms) {
    const bool fp8 = out_dtype == EP_FP8_E4M3;
    if (out_dtype != EP_BF16 && !fp8) return 0;
    if (hidden <= 0 || hidden % (fp8 ? 128 : 8) != 0) return 0;
    if (num_ranks < 1 || num_experts < num_ranks || num_experts % num_ranks != 0) return 0;
    if (num_topk < 1 || num_topk > EP_MAX_TOPK || num_topk > num_experts) return 0;
    if (!(hbm_gbs > 0.0) || !(sm_read_gbs > 0.0) || !(sm_write_gbs > 0.0) || device_sms < 1) return 0;
    // C(E - E/R, K) / C(E, K) = prod_{i<K} (E - E/R - i) / (E - i): the chance
    // that none of K distinct uniform experts lives on a given rank.
    const int others = num_experts - num_experts / num_ranks;
    double miss = 1.0;
    for (int i = 0; i < num_topk; ++i)
        miss *= others - i > 0 ? static_cast<double>(others - i) / (num_experts - i) : 0.0;
    const double g = num_ranks * (1.0 - miss);
    const double h = static_cast<double>(hidden);
    const double row = fp8 ? h + 4.0 * (h / 128.0) : 2.0 * h;
    const double read = is_combine ? g * 2.0 * h : 2.0 * h;
    const double write = is_combine ? 2.0 * h : g * row;
    const double per_byte = hbm_gbs / (read + write);
    const double n = std::max(per_byte * read / sm_read_gbs, per_byte * write / sm_write_gbs);
    int sms = std::max(4, static_cast<int>(std::ceil(n * 1.25)));
    sms += sms & 1;
    if (!prefer_overlap_with_compute) sms = std::max(sms, 64);
    return std::min(sms, device_sms);
}

int64_t ep_recv_capacity_bound(int num_tokens, int num_topk, int num_ranks) {
    if (num_tokens <= 0 || num_topk <= 0 || num_ranks <= 0) return 0;
    return static_cast<int64_t>(num_tokens) * (num_topk < num_ranks ? num_topk : num_ranks);
}

}  // extern "C"

namespace epg {

ep_status_t layout_params(const int64_t* topk_idx, int T, int K, int E, int R, int ranks_per_node,
                          int expert_alignment, const ep_layout_t* out, void* workspace, size_t ws_bytes,
                          int32_t* d_status, bool check_workspace, LayoutParams& p) {
    if (!out || !d_status) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (ranks_per_node < 0 || (ranks_per_node > 0 && R % ranks_per_node != 0))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (expert_alignment < 1) return EP_RET(EP_ERR_INVALID_ARG);
    if (!ok_ptr(out->num_tokens_per_rank) || !ok_ptr(out->num_tokens_per_expert) ||
        !ok_ptr(out->rank_offset) || !ok_ptr(out->expert_offset))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (T > 0 && (!ok_ptr(topk_idx) || !ok_ptr(out->is_token_in_rank) || !ok_ptr(out->dst_row)))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (out->num_tokens_per_node && !aligned16(out->num_tokens_per_node)) return EP_RET(EP_ERR_INVALID_ARG);
    if (out->src_dst_count && (!aligned16(out->src_dst_count) || T % R != 0)) return EP_RET(EP_ERR_INVALID_ARG);
    if (out->token_offset && !aligned16(out->token_offset)) return EP_RET(EP_ERR_INVALID_ARG);
    if (out->expanded_row && !aligned16(out->expanded_row)) return EP_RET(EP_ERR_INVALID_ARG);
    // node rows: node_offset and node_row together (node_row may be NULL, an
    // empty array, when there are no tokens)
    if (out->node_row && !out->node_offset) return EP_RET(EP_ERR_INVALID_ARG);
    if (out->node_offset && !out->node_row && T > 0) return EP_RET(EP_ERR_INVALID_ARG);
    if (out->node_offset && (ranks_per_node <= 0 || !ok_ptr(out->num_tokens_per_node) ||
                             !aligned16(out->node_row) || !aligned16(out->node_offset)))
        return EP_RET(EP_ERR_INVALID_ARG);
    const int nodes_ws = ranks_per_node > 0 ? R / ranks_per_node : 0;
    const epg::LayoutWorkspace w = epg::layout_workspace(T, E, R, nodes_ws);
    if (!check_workspace) return EP_OK;
    if (!ok_ptr(workspace) || ws_bytes < w.total) return EP_RET(EP_ERR_INVALID_ARG);

    p = epg::LayoutParams{};
    p.topk_idx = topk_idx;
    p.T = T;
    p.K = K;
    p.E = E;
    p.R = R;
    p.experts_per_rank = E / R;
    p.ranks_per_node = ranks_per_node;
    p.num_nodes = (ranks_per_node > 0 && out->num_tokens_per_node) ? R / ranks_per_node : 0;
    p.alignment = expert_alignment;
    p.num_tiles = (T + epg::kTileTokens - 1) / epg::kTileTokens;
    p.num_tokens_per_rank = out->num_tokens_per_rank;
    p.num_tokens_per_node = out->num_tokens_per_node;
    p.num_tokens_per_expert = out->num_tokens_per_expert;
    p.is_token_in_rank = out->is_token_in_rank;
    p.rank_offset = out->rank_offset;
    p.expert_offset = out->expert_offset;
    p.dst_row = out->dst_row;
    p.src_dst_count = out->src_dst_count;
    p.token_offset = out->token_offset;
    p.expanded_row = T > 0 ? out->expanded_row : nullptr;
    p.node_offset = out->node_offset;
    p.node_row = T > 0 ? out->node_row : nullptr;
    char* ws = static_cast<char*>(workspace);
    p.ws_rank = reinterpret_cast<int32_t*>(ws + w.off_rank);
    p.ws_expert = reinterpret_cast<int32_t*>(ws + w.off_expert);
    p.ws_node = reinterpret_cast<int32_t*>(ws + w.off_node);
    p.ws_bitmap = reinterpret_cast<uint32_t*>(ws + w.off_bitmap);
    p.status = d_status;
    return EP_OK;
}

}  // namespace epg

extern "C" {

ep_status_t ep_get_layout(const int64_t* topk_idx, int T, int K, int E, int R, int ranks_per_node,
                          int expert_alignment, const ep_layout_t* out, void* workspace,
                          size_t ws_bytes, int32_t* d_status, void* cuda_stream) {
    EP_DEBUG("ep_get_layout: T=%d K=%d E=%d R=%d ranks_per_node=%d alignment=%d%s%s",
             T, K, E, R, ranks_per_node, expert_alignment, out && out->expanded_row ? " expanded_row" : "",
             out && out->node_row ? " node_row" : "");
    epg::LayoutParams p{};
    const ep_status_t s = epg::layout_params(topk_idx, T, K, E, R, ranks_per_node, expert_alignment, out, workspace,
                                             ws_bytes, d_status, true, p);
    if (s != EP_OK) return s;
    const cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    if (epg::launch_layout(p, stream) != cudaSuccess) return EP_RET(EP_ERR_CUDA);
    // no tokens: the node-row kernels are not launched, node_offset is all zero
    if (T == 0 && out->node_offset &&
        cudaMemsetAsync(out->node_offset, 0, sizeof(int32_t) * (R / ranks_per_node + 1), stream) != cudaSuccess)
        return EP_RET(EP_ERR_CUDA);
    return EP_OK;
}

}  // extern "C"

namespace {

// A tag for the rows-ready signal, distinct for every call of the process:
// the splitmix64 output function (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", 2014), a bijection of 64-bit words,
// applied to a per-process offset plus an odd multiple of the call count.
uint64_t next_rows_tag() {
    static std::atomic<uint64_t> calls{0};
    static const uint64_t salt =
        static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) ^
        static_cast<uint64_t>(reinterpret_cast<uintptr_t>(&calls));
    uint64_t z = salt + 0x9e3779b97f4a7c15ull * (calls.fetch_add(1, std::memory_order_relaxed) + 1);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    z ^= z >> 31;
    return z != 0 ? z : 1;
}

// Shared by ep_dispatch and ep_layout_and_dispatch.  self_layout (few
// tokens, ep_layout_and_dispatch): no layout kernel has run; the dispatch
// kernel computes the rows itself and writes the layout arrays of `lp`.
ep_status_t dispatch_impl(const void* x, const int64_t* topk_idx, const float* topk_weights, int T, int H, int K,
                          int E, int R, const ep_layout_t* layout, int out_dtype, int64_t recv_capacity,
                          void* recv_x, float* recv_sf, int sf_col_major, int32_t* recv_topk_idx,
                          float* recv_topk_weights, int32_t* recv_src_idx, int num_sms, int32_t* d_status,
                          void* cuda_stream, const epg::LayoutParams* self_layout,
                          const epg::RowsSignal* rows = nullptr) {
    if (!layout || !d_status || num_sms < 0) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (H < 1) return EP_RET(EP_ERR_INVALID_ARG);
    if (out_dtype == EP_BF16) {
        if (H % 8 != 0) return EP_RET(EP_ERR_INVALID_ARG);
    } else if (out_dtype == EP_FP8_E4M3) {
        if (H % 128 != 0) return EP_RET(EP_ERR_INVALID_ARG);
        if (H > 65536) return EP_RET(EP_ERR_UNSUPPORTED);
    } else {
        return EP_RET(EP_ERR_INVALID_ARG);
    }
    if (recv_capacity < 0 || recv_capacity > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (static_cast<int64_t>(H) * 2 > UINT32_MAX / 2) return EP_RET(EP_ERR_UNSUPPORTED);
    if (T > 0 && (!ok_ptr(x) || !ok_ptr(topk_idx) || !ok_ptr(layout->dst_row)))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (recv_capacity > 0 && !ok_ptr(recv_x)) return EP_RET(EP_ERR_INVALID_ARG);
    if (out_dtype == EP_FP8_E4M3 && recv_capacity > 0 && !ok_ptr(recv_sf)) return EP_RET(EP_ERR_INVALID_ARG);
    if (recv_topk_weights && T > 0 && !ok_ptr(topk_weights)) return EP_RET(EP_ERR_INVALID_ARG);
    if ((recv_topk_idx && !aligned16(recv_topk_idx)) ||
        (recv_topk_weights && !aligned16(recv_topk_weights)) ||
        (recv_src_idx && !aligned16(recv_src_idx)))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (T == 0) return EP_OK;

    epg::DispatchParams p{};
    p.x = static_cast<const uint8_t*>(x);
    p.topk_idx = topk_idx;
    p.topk_weights = topk_weights;
    p.dst_row = layout->dst_row;
    p.token_offset = layout->token_offset;
    p.T = T;
    p.H = H;
    p.K = K;
    p.E = E;
    p.R = R;
    p.experts_per_rank = E / R;
    p.capacity = recv_capacity;
    p.recv_x = static_cast<uint8_t*>(recv_x);
    p.recv_sf = recv_sf;
    p.sf_col_major = sf_col_major ? 1 : 0;
    p.sf_stride = (recv_capacity + 3) / 4 * 4;
    p.recv_topk_idx = recv_topk_idx;
    p.recv_topk_weights = recv_topk_weights;
    p.recv_src_idx = recv_src_idx;
    p.num_sms = num_sms;
    p.status = d_status;
    if (self_layout) {
        p.self_route = 1;
        p.l_num_tokens_per_rank = self_layout->num_tokens_per_rank;
        p.l_num_tokens_per_node = self_layout->num_nodes > 0 ? self_layout->num_tokens_per_node : nullptr;
        p.l_num_tokens_per_expert = self_layout->num_tokens_per_expert;
        p.l_is_token_in_rank = self_layout->is_token_in_rank;
        p.l_rank_offset = self_layout->rank_offset;
        p.l_expert_offset = self_layout->expert_offset;
        p.l_dst_row = self_layout->dst_row;
        p.l_src_dst_count = self_layout->src_dst_count;
        p.l_token_offset = self_layout->token_offset;
        p.l_alignment = self_layout->alignment;
        p.l_ranks_per_node = self_layout->ranks_per_node;
        p.l_num_nodes = self_layout->num_nodes;
    }
    if (rows && rows->slots) {
        p.rows_ready = rows->slots;
        p.rows_tag = rows->tag;
        p.rows_tokens = rows->tokens;
        p.rows_slots = rows->count;
    }
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    const cudaError_t e = out_dtype == EP_BF16 ? epg::launch_dispatch_bf16(p, st)
                                               : epg::launch_dispatch_fp8(p, st);
    return e == cudaSuccess ? EP_OK : EP_RET(EP_ERR_CUDA);
}

}  // namespace

extern "C" {

ep_status_t ep_dispatch(const void* x, const int64_t* topk_idx, const float* topk_weights, int T,
                        int H, int K, int E, int R, const ep_layout_t* layout, int out_dtype,
                        int64_t recv_capacity, void* recv_x, float* recv_sf, int sf_col_major,
                        int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* recv_src_idx,
                        int num_sms, int32_t* d_status, void* cuda_stream) {
    EP_DEBUG("ep_dispatch: T=%d H=%d K=%d E=%d R=%d %s capacity=%lld sf_col_major=%d num_sms=%d",
             T, H, K, E, R, out_dtype == EP_FP8_E4M3 ? "fp8" : "bf16", static_cast<long long>(recv_capacity),
             sf_col_major, num_sms);
    return dispatch_impl(x, topk_idx, topk_weights, T, H, K, E, R, layout, out_dtype, recv_capacity, recv_x, recv_sf,
                         sf_col_major, recv_topk_idx, recv_topk_weights, recv_src_idx, num_sms, d_status, cuda_stream,
                         nullptr);
}

ep_status_t ep_layout_and_dispatch(const void* x, const int64_t* topk_idx, const float* topk_weights, int T, int H,
                                   int K, int E, int R, int ranks_per_node, int expert_alignment,
                                   const ep_layout_t* layout, void* workspace, size_t ws_bytes, int out_dtype,
                                   int64_t recv_capacity, void* recv_x, float* recv_sf, int sf_col_major,
                                   int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* recv_src_idx,
                                   int32_t* d_status, void* cuda_stream) {
    EP_DEBUG("ep_layout_and_dispatch: T=%d H=%d K=%d E=%d R=%d ranks_per_node=%d alignment=%d %s capacity=%lld",
             T, H, K, E, R, ranks_per_node, expert_alignment, out_dtype == EP_FP8_E4M3 ? "fp8" : "bf16",
             static_cast<long long>(recv_capacity));
    // the dispatch's host checks first, so that a rejected call launches nothing
    if (!layout || !d_status) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (H < 1 || (out_dtype != EP_BF16 && out_dtype != EP_FP8_E4M3)) return EP_RET(EP_ERR_INVALID_ARG);
    if (H % (out_dtype == EP_BF16 ? 8 : 128) != 0) return EP_RET(EP_ERR_INVALID_ARG);
    if (out_dtype == EP_FP8_E4M3 && H > 65536) return EP_RET(EP_ERR_UNSUPPORTED);
    if (recv_capacity < 0 || recv_capacity > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (static_cast<int64_t>(H) * 2 > UINT32_MAX / 2) return EP_RET(EP_ERR_UNSUPPORTED);
    if (T > 0 && (!ok_ptr(x) || !ok_ptr(topk_idx))) return EP_RET(EP_ERR_INVALID_ARG);
    if (recv_capacity > 0 && !ok_ptr(recv_x)) return EP_RET(EP_ERR_INVALID_ARG);
    if (out_dtype == EP_FP8_E4M3 && recv_capacity > 0 && !ok_ptr(recv_sf)) return EP_RET(EP_ERR_INVALID_ARG);
    if (recv_topk_weights && T > 0 && !ok_ptr(topk_weights)) return EP_RET(EP_ERR_INVALID_ARG);
    if ((recv_topk_idx && !aligned16(recv_topk_idx)) || (recv_topk_weights && !aligned16(recv_topk_weights)) ||
        (recv_src_idx && !aligned16(recv_src_idx)))
        return EP_RET(EP_ERR_INVALID_ARG);
    epg::LayoutParams lp{};
    s = epg::layout_params(topk_idx, T, K, E, R, ranks_per_node, expert_alignment, layout, workspace, ws_bytes,
                           d_status, true, lp);
    if (s != EP_OK) return s;
    // Few tokens: one kernel; its CTAs derive the rows themselves and write
    // the layout (expanded rows and node rows need the layout kernel).
    const bool one_kernel = T >= 1 && T <= epg::kSelfRouteMaxTokens && R <= 32 && K <= epg::kSelfRouteMaxTopk &&
                            E <= epg::kSelfRouteMaxExperts && !lp.expanded_row && !lp.node_row && !lp.node_offset;
    // Otherwise the layout kernel, and the dispatch waits for the rows-ready
    // signal of the cluster layout (where the dispatch kernel is one of the
    // two that read it) instead of the layout kernel's completion.
    epg::RowsSignal rows{};
    if (!one_kernel && T > 0 && epg::dispatch_reads_rows_signal(out_dtype == EP_FP8_E4M3) &&
        (reinterpret_cast<uintptr_t>(workspace) & 127u) == 0) {
        rows.slots = static_cast<uint64_t*>(workspace);
        rows.tag = next_rows_tag();
        rows.bytes = ws_bytes;
    }
    if (!one_kernel) {
        if (epg::launch_layout(lp, static_cast<cudaStream_t>(cuda_stream), &rows) != cudaSuccess)
            return EP_RET(EP_ERR_CUDA);
        if (T == 0 && layout->node_offset &&
            cudaMemsetAsync(layout->node_offset, 0, sizeof(int32_t) * (R / ranks_per_node + 1),
                            static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
            return EP_RET(EP_ERR_CUDA);
    }
    return dispatch_impl(x, topk_idx, topk_weights, T, H, K, E, R, layout, out_dtype, recv_capacity, recv_x, recv_sf,
                         sf_col_major, recv_topk_idx, recv_topk_weights, recv_src_idx, 0, d_status, cuda_stream,
                         one_kernel ? &lp : nullptr, &rows);
}

ep_status_t ep_dispatch_hierarchical(const void* x, const int64_t* topk_idx, const float* topk_weights, int T,
                                     int H, int K, int E, int R, int rpn, const ep_layout_t* layout,
                                     int out_dtype, int64_t node_capacity, void* node_x, float* node_sf,
                                     int32_t* node_src_idx, int64_t recv_capacity, void* recv_x, float* recv_sf,
                                     int sf_col_major, int32_t* recv_topk_idx, float* recv_topk_weights,
                                     int32_t* recv_src_idx, int32_t* d_status, void* cuda_stream) {
    EP_DEBUG("ep_dispatch_hierarchical: T=%d H=%d K=%d E=%d R=%d ranks_per_node=%d %s node_capacity=%lld capacity=%lld",
             T, H, K, E, R, rpn, out_dtype == EP_FP8_E4M3 ? "fp8" : "bf16", static_cast<long long>(node_capacity),
             static_cast<long long>(recv_capacity));
    if (!layout || !d_status) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (rpn < 1 || R % rpn != 0) return EP_RET(EP_ERR_INVALID_ARG);
    const bool fp8 = out_dtype == EP_FP8_E4M3;
    if (H < 1) return EP_RET(EP_ERR_INVALID_ARG);
    if (out_dtype == EP_BF16) {
        if (H % 8 != 0) return EP_RET(EP_ERR_INVALID_ARG);
    } else if (fp8) {
        if (H % 128 != 0) return EP_RET(EP_ERR_INVALID_ARG);
        if (H > 65536) return EP_RET(EP_ERR_UNSUPPORTED);
    } else {
        return EP_RET(EP_ERR_INVALID_ARG);
    }
    if (recv_capacity < 0 || recv_capacity > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (node_capacity < 0 || node_capacity > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (static_cast<int64_t>(H) * 2 > UINT32_MAX / 2) return EP_RET(EP_ERR_UNSUPPORTED);
    if (T > 0 && (!ok_ptr(x) || !ok_ptr(topk_idx) || !ok_ptr(layout->dst_row) || !ok_ptr(layout->node_row)))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (node_capacity > 0 && (!ok_ptr(node_x) || (fp8 && !ok_ptr(node_sf)))) return EP_RET(EP_ERR_INVALID_ARG);
    if (node_src_idx && !aligned16(node_src_idx)) return EP_RET(EP_ERR_INVALID_ARG);
    if (recv_capacity > 0 && !ok_ptr(recv_x)) return EP_RET(EP_ERR_INVALID_ARG);
    if (fp8 && recv_capacity > 0 && !ok_ptr(recv_sf)) return EP_RET(EP_ERR_INVALID_ARG);
    if (recv_topk_weights && T > 0 && !ok_ptr(topk_weights)) return EP_RET(EP_ERR_INVALID_ARG);
    if ((recv_topk_idx && !aligned16(recv_topk_idx)) || (recv_topk_weights && !aligned16(recv_topk_weights)) ||
        (recv_src_idx && !aligned16(recv_src_idx)))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (T == 0) return EP_OK;
    const int nodes = R / rpn;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);

    // stage 1: the ordinary dispatch with the node table as destinations
    epg::DispatchParams p{};
    p.x = static_cast<const uint8_t*>(x);
    p.topk_idx = topk_idx;
    p.topk_weights = topk_weights;
    p.dst_row = layout->node_row;
    p.T = T;
    p.H = H;
    p.K = K;
    p.E = E;
    p.R = nodes;
    p.experts_per_rank = E / R;
    p.capacity = node_capacity;
    p.recv_x = static_cast<uint8_t*>(node_x);
    p.recv_sf = node_sf;
    p.sf_col_major = 0;
    p.sf_stride = node_capacity;
    p.recv_src_idx = node_src_idx;
    p.status = d_status;
    cudaError_t e = fp8 ? epg::launch_dispatch_fp8(p, st) : epg::launch_dispatch_bf16(p, st);
    if (e != cudaSuccess) return EP_RET(EP_ERR_CUDA);

    // stage 2: node rows to the ranks of their node
    epg::HierParams h{};
    h.node_x = static_cast<const uint8_t*>(node_x);
    h.node_sf = node_sf;
    h.topk_idx = topk_idx;
    h.topk_weights = topk_weights;
    h.dst_row = layout->dst_row;
    h.node_row = layout->node_row;
    h.T = T;
    h.H = H;
    h.K = K;
    h.E = E;
    h.R = R;
    h.experts_per_rank = E / R;
    h.ranks_per_node = rpn;
    h.num_nodes = nodes;
    h.node_capacity = node_capacity;
    h.capacity = recv_capacity;
    h.recv_x = static_cast<uint8_t*>(recv_x);
    h.recv_sf = recv_sf;
    h.sf_col_major = sf_col_major ? 1 : 0;
    h.sf_stride = (recv_capacity + 3) / 4 * 4;
    h.recv_topk_idx = recv_topk_idx;
    h.recv_topk_weights = recv_topk_weights;
    h.recv_src_idx = recv_src_idx;
    h.status = d_status;
    return epg::launch_forward_scaleup(h, fp8, st) == cudaSuccess ? EP_OK : EP_RET(EP_ERR_CUDA);
}

ep_status_t ep_combine_hierarchical(const void* y, int64_t num_y_rows, const int64_t* topk_idx,
                                    const float* topk_weights, int T, int H, int K, int E, int R, int rpn,
                                    const ep_layout_t* layout, int64_t node_capacity, void* node_y, void* out,
                                    int32_t* d_status, void* cuda_stream) {
    EP_DEBUG("ep_combine_hierarchical: T=%d H=%d K=%d E=%d R=%d ranks_per_node=%d rows=%lld node_capacity=%lld %s",
             T, H, K, E, R, rpn, static_cast<long long>(num_y_rows), static_cast<long long>(node_capacity),
             topk_weights ? "weighted" : "unweighted");
    if (!layout || !d_status) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (rpn < 1 || R % rpn != 0) return EP_RET(EP_ERR_INVALID_ARG);
    if (H < 1 || H % 8 != 0) return EP_RET(EP_ERR_INVALID_ARG);
    if (num_y_rows < 0 || num_y_rows > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (node_capacity < 0 || node_capacity > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (num_y_rows > 0 && !ok_ptr(y)) return EP_RET(EP_ERR_INVALID_ARG);
    if (node_capacity > 0 && !ok_ptr(node_y)) return EP_RET(EP_ERR_INVALID_ARG);
    if (T > 0 && (!ok_ptr(out) || !ok_ptr(layout->dst_row) || !ok_ptr(layout->node_row)))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (topk_weights && T > 0 && (!ok_ptr(topk_weights) || !ok_ptr(topk_idx))) return EP_RET(EP_ERR_INVALID_ARG);
    if (T == 0) return EP_OK;
    const int nodes = R / rpn;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);

    // stage 1: per (token, node) partial sums of the node's ranks
    epg::HierParams h{};
    h.topk_idx = topk_idx;
    h.topk_weights = topk_weights;
    h.dst_row = layout->dst_row;
    h.node_row = layout->node_row;
    h.T = T;
    h.H = H;
    h.K = K;
    h.E = E;
    h.R = R;
    h.experts_per_rank = E / R;
    h.ranks_per_node = rpn;
    h.num_nodes = nodes;
    h.node_capacity = node_capacity;
    h.y = static_cast<const uint8_t*>(y);
    h.num_y_rows = num_y_rows;
    h.node_y = static_cast<uint8_t*>(node_y);
    h.status = d_status;
    if (epg::launch_reduce_scaleup(h, topk_weights != nullptr, st) != cudaSuccess) return EP_RET(EP_ERR_CUDA);

    // stage 2: the ordinary unweighted combine over the node rows
    epg::CombineParams p{};
    p.y = static_cast<const uint8_t*>(node_y);
    p.num_y_rows = node_capacity;
    p.topk_idx = topk_idx;
    p.dst_row = layout->node_row;
    p.T = T;
    p.H = H;
    p.K = K;
    p.E = E;
    p.R = nodes;
    p.experts_per_rank = E / R;
    p.out = static_cast<uint8_t*>(out);
    p.status = d_status;
    return epg::launch_combine(p, false, st) == cudaSuccess ? EP_OK : EP_RET(EP_ERR_CUDA);
}

ep_status_t ep_combine(const void* y, int64_t num_y_rows, const int64_t* topk_idx,
                       const float* topk_weights, int T, int H, int K, int E, int R,
                       const ep_layout_t* layout, void* out, int num_sms, int32_t* d_status,
                       void* cuda_stream) {
    EP_DEBUG("ep_combine: T=%d H=%d K=%d E=%d R=%d rows=%lld %s num_sms=%d",
             T, H, K, E, R, static_cast<long long>(num_y_rows), topk_weights ? "weighted" : "unweighted", num_sms);
    if (!layout || !d_status || num_sms < 0) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (H < 1 || H % 8 != 0) return EP_RET(EP_ERR_INVALID_ARG);
    if (num_y_rows < 0 || num_y_rows > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (num_y_rows > 0 && !ok_ptr(y)) return EP_RET(EP_ERR_INVALID_ARG);
    if (T > 0 && (!ok_ptr(out) || !ok_ptr(layout->dst_row))) return EP_RET(EP_ERR_INVALID_ARG);
    if (topk_weights && T > 0 && (!ok_ptr(topk_weights) || !ok_ptr(topk_idx))) return EP_RET(EP_ERR_INVALID_ARG);
    if (T == 0) return EP_OK;

    epg::CombineParams p{};
    p.y = static_cast<const uint8_t*>(y);
    p.num_y_rows = num_y_rows;
    p.topk_idx = topk_idx;
    p.topk_weights = topk_weights;
    p.dst_row = layout->dst_row;
    p.T = T;
    p.H = H;
    p.K = K;
    p.E = E;
    p.R = R;
    p.experts_per_rank = E / R;
    p.out = static_cast<uint8_t*>(out);
    p.num_sms = num_sms;
    p.status = d_status;
    const cudaError_t e =
        epg::launch_combine(p, topk_weights != nullptr, static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? EP_OK : EP_RET(EP_ERR_CUDA);
}

int64_t ep_expanded_capacity_bound(int num_tokens, int num_topk, int num_experts, int expert_alignment) {
    if (num_tokens < 0 || num_topk < 0 || num_experts < 0 || expert_alignment < 1) return 0;
    return static_cast<int64_t>(num_tokens) * num_topk + static_cast<int64_t>(num_experts) * (expert_alignment - 1);
}

ep_status_t ep_dispatch_expanded(const void* x, const int64_t* topk_idx, const float* topk_weights, int T,
                                 int H, int K, int E, int R, const ep_layout_t* layout, int out_dtype,
                                 int64_t recv_capacity, void* recv_x, float* recv_sf, int sf_col_major,
                                 int32_t* recv_src_idx, float* recv_weight, int num_sms, int32_t* d_status,
                                 void* cuda_stream) {
    EP_DEBUG("ep_dispatch_expanded: T=%d H=%d K=%d E=%d R=%d %s capacity=%lld sf_col_major=%d num_sms=%d",
             T, H, K, E, R, out_dtype == EP_FP8_E4M3 ? "fp8" : "bf16", static_cast<long long>(recv_capacity),
             sf_col_major, num_sms);
    if (!layout || !d_status || num_sms < 0) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (H < 1) return EP_RET(EP_ERR_INVALID_ARG);
    if (out_dtype == EP_BF16) {
        if (H % 8 != 0) return EP_RET(EP_ERR_INVALID_ARG);
    } else if (out_dtype == EP_FP8_E4M3) {
        if (H % 128 != 0) return EP_RET(EP_ERR_INVALID_ARG);
        if (H > 65536) return EP_RET(EP_ERR_UNSUPPORTED);
    } else {
        return EP_RET(EP_ERR_INVALID_ARG);
    }
    if (recv_capacity < 0 || recv_capacity > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (static_cast<int64_t>(H) * 2 > UINT32_MAX / 2) return EP_RET(EP_ERR_UNSUPPORTED);
    if (T > 0 && (!ok_ptr(x) || !ok_ptr(layout->expanded_row))) return EP_RET(EP_ERR_INVALID_ARG);
    if (recv_capacity > 0 && !ok_ptr(recv_x)) return EP_RET(EP_ERR_INVALID_ARG);
    if (out_dtype == EP_FP8_E4M3 && recv_capacity > 0 && !ok_ptr(recv_sf)) return EP_RET(EP_ERR_INVALID_ARG);
    if (recv_weight && T > 0 && !ok_ptr(topk_weights)) return EP_RET(EP_ERR_INVALID_ARG);
    if ((recv_src_idx && !aligned16(recv_src_idx)) || (recv_weight && !aligned16(recv_weight)))
        return EP_RET(EP_ERR_INVALID_ARG);
    if (T == 0) return EP_OK;

    epg::DispatchParams p{};
    p.x = static_cast<const uint8_t*>(x);
    p.topk_idx = topk_idx;
    p.topk_weights = topk_weights;
    p.expanded_row = layout->expanded_row;
    p.T = T;
    p.H = H;
    p.K = K;
    p.E = E;
    p.R = R;
    p.experts_per_rank = E / R;
    p.capacity = recv_capacity;
    p.recv_x = static_cast<uint8_t*>(recv_x);
    p.recv_sf = recv_sf;
    p.sf_col_major = sf_col_major ? 1 : 0;
    p.sf_stride = (recv_capacity + 3) / 4 * 4;
    p.recv_src_idx = recv_src_idx;
    p.recv_weight = recv_weight;
    p.num_sms = num_sms;
    p.status = d_status;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    const cudaError_t e = out_dtype == EP_BF16 ? epg::launch_dispatch_bf16(p, st)
                                               : epg::launch_dispatch_fp8(p, st);
    return e == cudaSuccess ? EP_OK : EP_RET(EP_ERR_CUDA);
}

ep_status_t ep_combine_expanded(const void* y, int64_t num_y_rows, const float* topk_weights, int T, int H,
                                int K, int E, int R, const ep_layout_t* layout, void* out, int num_sms,
                                int32_t* d_status, void* cuda_stream) {
    EP_DEBUG("ep_combine_expanded: T=%d H=%d K=%d E=%d R=%d rows=%lld %s num_sms=%d",
             T, H, K, E, R, static_cast<long long>(num_y_rows), topk_weights ? "weighted" : "unweighted", num_sms);
    if (!layout || !d_status || num_sms < 0) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (H < 1 || H % 8 != 0) return EP_RET(EP_ERR_INVALID_ARG);
    if (num_y_rows < 0 || num_y_rows > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (num_y_rows > 0 && !ok_ptr(y)) return EP_RET(EP_ERR_INVALID_ARG);
    if (T > 0 && (!ok_ptr(out) || !ok_ptr(layout->expanded_row))) return EP_RET(EP_ERR_INVALID_ARG);
    if (topk_weights && T > 0 && !ok_ptr(topk_weights)) return EP_RET(EP_ERR_INVALID_ARG);
    if (T == 0) return EP_OK;

    epg::CombineParams p{};
    p.y = static_cast<const uint8_t*>(y);
    p.num_y_rows = num_y_rows;
    p.topk_weights = topk_weights;
    p.expanded_row = layout->expanded_row;
    p.T = T;
    p.H = H;
    p.K = K;
    p.E = E;
    p.R = R;
    p.experts_per_rank = E / R;
    p.out = static_cast<uint8_t*>(out);
    p.num_sms = num_sms;
    p.status = d_status;
    const cudaError_t e =
        epg::launch_combine(p, topk_weights != nullptr, static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? EP_OK : EP_RET(EP_ERR_CUDA);
}

ep_status_t ep_combine_topk_weights(const float* recv_topk_weights, int64_t num_rows, int T, int K, int E,
                                   int R, const ep_layout_t* layout, float* combined_topk_weights,
                                   int32_t* d_status, void* cuda_stream) {
    EP_DEBUG("ep_combine_topk_weights: T=%d K=%d E=%d R=%d rows=%lld", T, K, E, R, static_cast<long long>(num_rows));
    if (!layout || !d_status) return EP_RET(EP_ERR_INVALID_ARG);
    ep_status_t s = check_shape(T, K, E, R);
    if (s != EP_OK) return s;
    if (num_rows < 0 || num_rows > INT32_MAX) return EP_RET(EP_ERR_INVALID_ARG);
    if (num_rows > 0 && !ok_ptr(recv_topk_weights)) return EP_RET(EP_ERR_INVALID_ARG);
    if (T > 0 && (!ok_ptr(combined_topk_weights) || !ok_ptr(layout->dst_row))) return EP_RET(EP_ERR_INVALID_ARG);
    if (T == 0) return EP_OK;
    epg::CombineWeightsParams p{};
    p.recv_topk_weights = recv_topk_weights;
    p.num_rows = num_rows;
    p.dst_row = layout->dst_row;
    p.T = T;
    p.K = K;
    p.R = R;
    p.combined = combined_topk_weights;
    p.status = d_status;
    return epg::launch_combine_topk_weights(p, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
               ? EP_OK
               : EP_ERR_CUDA;
}

ep_status_t ep_accumulate_expert_stats(const ep_layout_t* layout, int E, int64_t* stats, void* cuda_stream) {
    EP_DEBUG("ep_accumulate_expert_stats: E=%d", E);
    if (!layout || E < 1) return EP_RET(EP_ERR_INVALID_ARG);
    if (E > EP_MAX_EXPERTS) return EP_RET(EP_ERR_UNSUPPORTED);
    if (!ok_ptr(layout->num_tokens_per_expert) || !ok_ptr(stats)) return EP_RET(EP_ERR_INVALID_ARG);
    return epg::launch_accumulate_expert_stats(layout->num_tokens_per_expert, E, stats,
                                               static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess
               ? EP_OK
               : EP_ERR_CUDA;
}

const char* ep_status_string(int32_t status) {
    static const char* const kNames[7] = {"invalid_arg", "unsupported", "invalid_index", "capacity",
                                          "timeout",     "cuda",        "out_of_bounds"};
    static std::string table[128];
    static std::once_flag once;
    std::call_once(once, [] {
        table[0] = "ok";
        for (int v = 1; v < 128; ++v) {
            std::string sname;
            for (int b = 0; b < 7; ++b)
                if (v & (1 << b)) {
                    if (!sname.empty()) sname += "|";
                    sname += kNames[b];
                }
            table[v] = sname;
        }
    });
    if (status < 0 || status >= 128) return "unknown";
    return table[status].c_str();
}

}  // extern "C"
