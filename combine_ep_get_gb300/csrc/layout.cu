// Routing layout on the GPU: per-rank / per-expert / per-node receive counts,
// token->rank membership, and deterministic receive rows.
//
// Outputs follow "DeepEP Symmetric Memory" section 6.1 (per-rank and
// per-expert prefix sums of receive counts, a destination slot per token,
// expert_alignment) and section 7.3 (receive counts per rank and per local
// expert).  Receive order inside a rank is ascending token index, so every
// output is a pure function of topk_idx: no atomic decides an order.
//
// Three launches over tiles of 256 tokens:
//   1. count:  per tile, a shared-memory membership bitmap [R][8 words]
//              (bit t of rank r set when token t has an expert on r), built
//              from coalesced top-k loads with shared atomics; per-tile rank,
//              expert and node counts go to the workspace, columns by tile.
//   2. scan:   one warp per rank / expert / node column: the exclusive prefix
//              over tiles (ranks) and the column totals (the count outputs).
//   3. rows:   per tile, rank_offset by a block scan of the rank totals, then
//              dst_row and is_token_in_rank for the tile's contiguous [256,R]
//              block: base of (rank, tile) + popc of the bitmap below the
//              token.  Block 0 also writes rank_offset and expert_offset.
#include "ep_internal.cuh"

namespace epg {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) layout_count_kernel(const LayoutParams p) {
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ int s_bad;
    const int R = p.R;
    uint32_t* s_bm = smem;                                       // [R][kTileWords]
    uint32_t* s_bm_node = s_bm + R * kTileWords;                 // [num_nodes][kTileWords]
    int* s_hist = reinterpret_cast<int*>(s_bm_node + p.num_nodes * kTileWords);  // [E]
    const int tile = blockIdx.x;
    const int n_words = R * kTileWords + p.num_nodes * kTileWords + p.E;

    // The src_dst_count output is accumulated by the rows kernel: zero it here.
    if (p.src_dst_count) {
        const int nn = R * R;
        for (int i = blockIdx.x * kThreads + threadIdx.x; i < nn; i += gridDim.x * kThreads)
            p.src_dst_count[i] = 0;
    }
    if (tile >= p.num_tiles) return;

    for (int i = threadIdx.x; i < n_words; i += kThreads) smem[i] = 0u;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();

    const int t0 = tile * kTileTokens;
    const int nt = min(kTileTokens, p.T - t0);
    const int n_entries = nt * p.K;
    const int64_t* src = p.topk_idx + static_cast<int64_t>(t0) * p.K;
    bool bad = false;
    for (int i = threadIdx.x; i < n_entries; i += kThreads) {
        const int64_t e = src[i];
        if (e == -1) continue;
        if (e < -1 || e >= p.E) { bad = true; continue; }
        const int tl = i / p.K;
        const int r = static_cast<int>(e) / p.experts_per_rank;
        const uint32_t bit = 1u << (tl & 31);
        atomicAdd(&s_hist[e], 1);
        atomicOr(&s_bm[r * kTileWords + (tl >> 5)], bit);
        if (p.num_nodes) atomicOr(&s_bm_node[(r / p.ranks_per_node) * kTileWords + (tl >> 5)], bit);
    }
    if (bad) s_bad = 1;
    __syncthreads();

    uint32_t* g_bm = p.ws_bitmap + static_cast<size_t>(tile) * R * kTileWords;
    for (int i = threadIdx.x; i < R * kTileWords; i += kThreads) g_bm[i] = s_bm[i];
    for (int r = threadIdx.x; r < R; r += kThreads) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kTileWords; ++w) c += __popc(s_bm[r * kTileWords + w]);
        p.ws_rank[static_cast<size_t>(r) * p.num_tiles + tile] = c;
    }
    for (int e = threadIdx.x; e < p.E; e += kThreads)
        p.ws_expert[static_cast<size_t>(e) * p.num_tiles + tile] = s_hist[e];
    for (int n = threadIdx.x; n < p.num_nodes; n += kThreads) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kTileWords; ++w) c += __popc(s_bm_node[n * kTileWords + w]);
        p.ws_node[static_cast<size_t>(n) * p.num_tiles + tile] = c;
    }
    if (threadIdx.x == 0 && s_bad) atomicOr(p.status, EP_ERR_INVALID_INDEX);
}

// One warp per column: ranks [0,R), experts [R, R+E), nodes [R+E, R+E+nodes).
__global__ void __launch_bounds__(kThreads) layout_scan_kernel(const LayoutParams p) {
    const int col = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int n_cols = p.R + p.E + p.num_nodes;
    if (col >= n_cols) return;
    int32_t* row;
    int32_t* total;
    bool scan = false;
    if (col < p.R) {
        row = p.ws_rank + static_cast<size_t>(col) * p.num_tiles;
        total = p.num_tokens_per_rank + col;
        scan = true;
    } else if (col < p.R + p.E) {
        const int e = col - p.R;
        row = p.ws_expert + static_cast<size_t>(e) * p.num_tiles;
        total = p.num_tokens_per_expert + e;
    } else {
        const int n = col - p.R - p.E;
        row = p.ws_node + static_cast<size_t>(n) * p.num_tiles;
        total = p.num_tokens_per_node + n;
    }
    int carry = 0;
    for (int base = 0; base < p.num_tiles; base += 32) {
        const int i = base + lane;
        const int v = i < p.num_tiles ? row[i] : 0;
        const int incl = warp_inclusive_scan(v);
        if (scan && i < p.num_tiles) row[i] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) *total = carry;
}

// Exclusive scan over n values get(i); put(i, prefix) for i in [0, n] with
// put(n, total).  Called by all kThreads threads; s_warp holds 8 ints.
template <class Get, class Put>
__device__ void block_exclusive_scan(int n, Get get, Put put, int* s_warp) {
    const int tid = threadIdx.x;
    const int per = (n + kThreads - 1) / kThreads;
    const int begin = min(n, tid * per);
    const int end = min(n, begin + per);
    int local = 0;
    for (int i = begin; i < end; ++i) local += get(i);
    const int incl = warp_inclusive_scan(local);
    const int lane = tid & 31, warp = tid >> 5;
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const int s = s_warp[w];
        if (w < warp) before += s;
        total += s;
    }
    int run = before + incl - local;
    for (int i = begin; i < end; ++i) {
        put(i, run);
        run += get(i);
    }
    if (tid == 0) put(n, total);
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) layout_rows_kernel(const LayoutParams p) {
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ int s_warp[kThreads / 32];
    const int R = p.R;
    int* s_base = reinterpret_cast<int*>(smem);                 // [R+1]
    uint32_t* s_bm = smem + (R + 1);                             // [R][kTileWords]
    int* s_wpre = reinterpret_cast<int*>(s_bm + R * kTileWords);  // [R][kTileWords]
    const int tile = blockIdx.x;

    const int32_t* cnt = p.num_tokens_per_rank;
    block_exclusive_scan(R, [&](int i) { return cnt[i]; }, [&](int i, int v) { s_base[i] = v; },
                         s_warp);
    if (tile == 0) {
        for (int i = threadIdx.x; i <= R; i += kThreads) p.rank_offset[i] = s_base[i];
        const int a = p.alignment;
        const int32_t* ce = p.num_tokens_per_expert;
        int32_t* eo = p.expert_offset;
        block_exclusive_scan(
            p.E, [&](int i) { return (ce[i] + a - 1) / a * a; }, [&](int i, int v) { eo[i] = v; },
            s_warp);
    }
    if (tile >= p.num_tiles) return;

    for (int r = threadIdx.x; r < R; r += kThreads)
        s_base[r] += p.ws_rank[static_cast<size_t>(r) * p.num_tiles + tile];
    const uint32_t* g_bm = p.ws_bitmap + static_cast<size_t>(tile) * R * kTileWords;
    for (int i = threadIdx.x; i < R * kTileWords; i += kThreads) s_bm[i] = g_bm[i];
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += kThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kTileWords; ++w) {
            s_wpre[r * kTileWords + w] = run;
            run += __popc(s_bm[r * kTileWords + w]);
        }
    }
    __syncthreads();

    const int t0 = tile * kTileTokens;
    const int nt = min(kTileTokens, p.T - t0);
    const int n_el = nt * R;
    int32_t* drow = p.dst_row + static_cast<size_t>(t0) * R;
    uint8_t* inr = p.is_token_in_rank + static_cast<size_t>(t0) * R;
    for (int j = threadIdx.x; j < n_el; j += kThreads) {
        const int tl = j / R;
        const int r = j - tl * R;
        const int w = tl >> 5;
        const uint32_t word = s_bm[r * kTileWords + w];
        const uint32_t b = static_cast<uint32_t>(tl & 31);
        const bool in = (word >> b) & 1u;
        drow[j] = in ? s_base[r] + s_wpre[r * kTileWords + w] + __popc(word & ((1u << b) - 1u)) : -1;
        inr[j] = in ? 1 : 0;
    }

    // src_dst_count[s][r]: tokens of source rank s (tokens [s*T/R, (s+1)*T/R)) in rank r.
    if (p.src_dst_count) {
        const int ts = p.T / R;
        const int s_lo = t0 / ts;
        const int s_hi = (t0 + nt - 1) / ts;
        const int n_pairs = (s_hi - s_lo + 1) * R;
        for (int q = threadIdx.x; q < n_pairs; q += kThreads) {
            const int s = s_lo + q / R;
            const int r = q - (q / R) * R;
            const int a = max(t0, s * ts) - t0;
            const int b = min(t0 + nt, (s + 1) * ts) - t0;
            int c = 0;
            for (int w = a >> 5; w <= (b - 1) >> 5; ++w) {
                const int lo = max(a - w * 32, 0);
                const int hi = min(b - w * 32, 32);
                const uint32_t upper = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
                const uint32_t mask = upper & ~((1u << lo) - 1u);
                c += __popc(s_bm[r * kTileWords + w] & mask);
            }
            if (c) atomicAdd(&p.src_dst_count[s * R + r], c);
        }
    }
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

LayoutWorkspace layout_workspace(int T, int E, int R, int num_nodes) {
    const size_t tiles = (static_cast<size_t>(T) + kTileTokens - 1) / kTileTokens;
    LayoutWorkspace w;
    size_t off = 0;
    w.off_rank = off;
    off = align_up(off + 4 * static_cast<size_t>(R) * tiles, 256);
    w.off_expert = off;
    off = align_up(off + 4 * static_cast<size_t>(E) * tiles, 256);
    w.off_node = off;
    off = align_up(off + 4 * static_cast<size_t>(num_nodes) * tiles, 256);
    w.off_bitmap = off;
    off = align_up(off + 4 * static_cast<size_t>(R) * kTileWords * tiles, 256);
    w.total = off < 16 ? 16 : off;
    return w;
}

cudaError_t launch_layout(const LayoutParams& p, cudaStream_t stream) {
    const DeviceInfo& di = device_info();
    const size_t smem_count =
        4 * (static_cast<size_t>(p.R) * kTileWords + static_cast<size_t>(p.num_nodes) * kTileWords + p.E);
    const size_t smem_rows = 4 * (static_cast<size_t>(p.R) + 1 + 2 * static_cast<size_t>(p.R) * kTileWords);
    static thread_local int configured_device = -1;
    if (configured_device != di.device) {
        // Worst case over the supported limits (R = 1024, E = 2048): < 80 KB.
        const int cap = di.max_smem_optin < 100 * 1024 ? di.max_smem_optin : 100 * 1024;
        cudaError_t e = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(layout_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
        if (e != cudaSuccess) return e;
        configured_device = di.device;
    }
    const int grid_tiles = p.num_tiles > 0 ? p.num_tiles : 1;
    layout_count_kernel<<<grid_tiles, kThreads, smem_count, stream>>>(p);
    const int n_cols = p.R + p.E + p.num_nodes;
    const int scan_blocks = (n_cols * 32 + kThreads - 1) / kThreads;
    layout_scan_kernel<<<scan_blocks, kThreads, 0, stream>>>(p);
    layout_rows_kernel<<<grid_tiles, kThreads, smem_rows, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace epg
