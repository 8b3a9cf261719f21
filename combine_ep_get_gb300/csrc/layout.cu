// Routing layout on the GPU: per-rank / per-expert / per-node receive counts,
// token->rank membership, and deterministic receive rows.
//
// Outputs follow "DeepEP Symmetric Memory" section 6.1 (per-rank and
// per-expert prefix sums of receive counts, a destination slot per token,
// expert_alignment) and section 7.3 (receive counts per rank and per local
// expert).  Receive order inside a rank is ascending token index, so every
// output is a pure function of topk_idx: no atomic decides an order.
//
// Few tokens (T <= 1024, R <= 32, K <= 16): one CTA, no cluster (see
// layout_small_kernel), since at that size the cluster's fixed phases cost more
// than the work.
//
// Main path (T * R <= 2^19): ONE launch of one thread-block cluster (up to
// 16 CTAs of 1024 threads, one per SM).  CTA c owns a contiguous token range;
// it builds the membership bitmaps [words][R] and the expert histogram of its
// range in shared memory, then after a hardware cluster barrier every CTA
// reads the other CTAs' per-rank counts through distributed shared memory to
// get its base row per rank (rank_offset + earlier CTAs); CTA 0 writes the
// rank counts and offsets and the last CTA gathers the expert / node counts
// and writes them with the expert offsets.  Each CTA then writes dst_row and
// is_token_in_rank for its range with 16-byte stores (behind
// ep_layout_and_dispatch it then publishes a rows-ready tag in its workspace
// line, on which the dispatch's first wave starts), then its token offsets
// and src_dst_count; a closing cluster barrier keeps every CTA's shared
// memory alive for the other CTAs' remote reads.  No global-memory
// synchronisation and no spin inside the kernel.
//
// Fallback (T * R > 2^19, or a CTA's bitmaps would not fit in shared memory):
// three launches over tiles of 256 tokens:
//   1. count:  per tile, a shared-memory membership bitmap [8 words][R]
//              (bit t of rank r set when token t has an expert on r), built
//              from coalesced top-k loads with shared atomics; per-tile rank,
//              expert and node counts go to the workspace, columns by tile.
//   2. scan:   one warp per rank / expert / node column: the exclusive prefix
//              over tiles (ranks) and the column totals (the count outputs).
//   3. rows:   per tile, rank_offset by a block scan of the rank totals, then
//              dst_row and is_token_in_rank for the tile's contiguous [256,R]
//              block: base of (rank, tile) + popc of the bitmap below the
//              token.  Block 0 also writes rank_offset and expert_offset.
#include <cooperative_groups.h>

#include "ep_internal.cuh"

namespace epg {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kStageUnroll = 8;   // global loads in flight per thread when staging into shared memory

// Sum of v over the block (blockDim a multiple of 32, at most 1024); s_red
// holds 33 ints.  Every thread gets the total.
__device__ int block_sum(int v, int* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int x = lane < n_warps ? s_red[lane] : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) s_red[32] = x;
    }
    __syncthreads();
    const int total = s_red[32];
    __syncthreads();
    return total;
}


__global__ void __launch_bounds__(kThreads) layout_count_kernel(const LayoutParams p) {
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ int s_bad;
    const int R = p.R;
    uint32_t* s_bm = smem;                                       // [kTileWords][R]
    uint32_t* s_bm_node = s_bm + R * kTileWords;                 // [kTileWords][num_nodes]
    int* s_hist = reinterpret_cast<int*>(s_bm_node + p.num_nodes * kTileWords);  // [E]
    const int tile = blockIdx.x;
    const int n_words = R * kTileWords + p.num_nodes * kTileWords + p.E;
    pdl_wait();   // first: the previous kernel may write topk_idx or read our outputs

    // The src_dst_count output is accumulated by the rows kernel: zero it here.
    if (p.src_dst_count) {
        const int nn = R * R;
        for (int i = blockIdx.x * kThreads + threadIdx.x; i < nn; i += gridDim.x * kThreads)
            if (EP_IN(i, nn)) p.src_dst_count[i] = 0;
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
    for (int base = 0; base < n_entries; base += kUnroll * kThreads) {
        int64_t e[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * kThreads + threadIdx.x;
            e[u] = (i < n_entries && EP_IN(static_cast<int64_t>(t0) * p.K + i, static_cast<int64_t>(p.T) * p.K))
                       ? src[i] : -1;     // all loads in flight before any use
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * kThreads + threadIdx.x;
            if (e[u] == -1) continue;
            if (e[u] < -1 || e[u] >= p.E) { bad = true; continue; }
            const int tl = i / p.K;
            const int r = static_cast<int>(e[u]) / p.experts_per_rank;
            const uint32_t bit = 1u << (tl & 31);
            atomicAdd(&s_hist[e[u]], 1);
            atomicOr(&s_bm[(tl >> 5) * R + r], bit);
            if (p.num_nodes) atomicOr(&s_bm_node[(tl >> 5) * p.num_nodes + r / p.ranks_per_node], bit);
        }
    }
    if (bad) s_bad = 1;
    __syncthreads();

    const int64_t bm0 = static_cast<int64_t>(tile) * R * kTileWords;
    const int64_t n_bm = static_cast<int64_t>(p.num_tiles) * R * kTileWords;
    uint32_t* g_bm = p.ws_bitmap + bm0;
    for (int i = threadIdx.x; i < R * kTileWords; i += kThreads)
        if (EP_IN(bm0 + i, n_bm)) g_bm[i] = s_bm[i];
    for (int r = threadIdx.x; r < R; r += kThreads) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kTileWords; ++w) c += __popc(s_bm[w * R + r]);
        const int64_t wi = static_cast<int64_t>(r) * p.num_tiles + tile;
        if (EP_IN(wi, static_cast<int64_t>(R) * p.num_tiles)) p.ws_rank[wi] = c;
    }
    for (int e = threadIdx.x; e < p.E; e += kThreads) {
        const int64_t wi = static_cast<int64_t>(e) * p.num_tiles + tile;
        if (EP_IN(wi, static_cast<int64_t>(p.E) * p.num_tiles)) p.ws_expert[wi] = s_hist[e];
    }
    for (int n = threadIdx.x; n < p.num_nodes; n += kThreads) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kTileWords; ++w) c += __popc(s_bm_node[w * p.num_nodes + n]);
        const int64_t wi = static_cast<int64_t>(n) * p.num_tiles + tile;
        if (EP_IN(wi, static_cast<int64_t>(p.num_nodes) * p.num_tiles)) p.ws_node[wi] = c;
    }
    if (threadIdx.x == 0 && s_bad) atomicOr(p.status, EP_ERR_INVALID_INDEX);
}

// One warp per column: ranks [0,R), experts [R, R+E), nodes [R+E, R+E+nodes).
__global__ void __launch_bounds__(kThreads) layout_scan_kernel(const LayoutParams p) {
    pdl_wait();
    const int col = (blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int n_cols = p.R + p.E + p.num_nodes;
    if (col >= n_cols) return;
    int32_t* row;
    int32_t* total;
    bool scan = false;
    // the column's workspace row and total stay inside their arrays
    if (!EP_IN(col, n_cols)) return;
    if (col < p.R) {
        row = p.ws_rank + static_cast<size_t>(col) * p.num_tiles;
        total = p.num_tokens_per_rank + col;
        scan = true;
    } else if (col < p.R + p.E) {
        const int e = col - p.R;
        row = p.ws_expert + static_cast<size_t>(e) * p.num_tiles;
        total = p.num_tokens_per_expert + e;
        scan = p.expanded_row != nullptr;   // tile prefix per expert for the expanded rows
    } else {
        const int n = col - p.R - p.E;
        row = p.ws_node + static_cast<size_t>(n) * p.num_tiles;
        total = p.num_tokens_per_node + n;
        scan = p.node_row != nullptr;        // tile prefix per node for the node rows
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

// Per-thread register slices for the rows kernel's scans: thread tid holds
// elements tid * per + j (j < per, per = ceil(n / kThreads)) of an n-vector.
constexpr int kMaxRankSlice = (EP_MAX_RANKS + kThreads - 1) / kThreads;
constexpr int kMaxExpertSlice = (EP_MAX_EXPERTS + kThreads - 1) / kThreads;

// v[j] = enable ? get(tid * per + j) : 0 for the thread's slice, all loads
// issued before any use.
template <int kMax, class Get>
__device__ __forceinline__ void load_slice(int (&v)[kMax], int n, int per, bool enable, Get get) {
#pragma unroll
    for (int j = 0; j < kMax; ++j) {
        const int i = static_cast<int>(threadIdx.x) * per + j;
        v[j] = (enable && j < per && i < n) ? get(i) : 0;
    }
}

// Exclusive scan of an n-vector held in register slices (see load_slice):
// out[j] = sum of the elements before element tid * per + j.  Returns the
// total.  Called by all kThreads threads; s_warp holds 8 ints.
template <int kMax>
__device__ int block_exclusive_scan_slice(const int (&v)[kMax], int (&out)[kMax], int per, int* s_warp) {
    const int tid = threadIdx.x;
    int local = 0;
#pragma unroll
    for (int j = 0; j < kMax; ++j) local += j < per ? v[j] : 0;
    const int incl = warp_inclusive_scan(local);
    const int lane = tid & 31, warp = tid >> 5;
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const int x = s_warp[w];
        if (w < warp) before += x;
        total += x;
    }
    int run = before + incl - local;
#pragma unroll
    for (int j = 0; j < kMax; ++j) {
        out[j] = run;
        run += j < per ? v[j] : 0;
    }
    __syncthreads();
    return total;
}

// The lanes of the warp whose key equals this lane's (what the warp match
// instruction returns), through a per-(warp, key) word in shared memory: each
// lane ORs its bit in, the warp reads the word back, and the group's first
// lane clears it.  kb: this warp's [E] words, zero on entry and left zero.
// Negative keys are unique per lane.  When every warp of an SM ranks at once
// the match instruction serialises (~2 us for two passes over 64 chunks);
// a shared atomic, a load and a store per lane do not.
__device__ __forceinline__ unsigned match_key(int key, uint32_t* kb, int lane) {
    if (key >= 0) atomicOr(&kb[key], 1u << lane);
    __syncwarp();
    const unsigned g = key >= 0 ? kb[key] : (1u << lane);
    __syncwarp();
    if (key >= 0 && lane == __ffs(g) - 1) kb[key] = 0u;
    return g;
}

// Ranks entries [0, n_ent) per expert in index order: entry i with key
// e >= 0 (s_key[i]; negative keys are unique per lane and never match) gets
// out[i] = s_eb[e] + (entries of e before i), else -1.  Warps 0..nw-1 each
// rank a contiguous slice of 32-entry chunks twice around per-(warp, expert)
// bases in s_wc [nw][E]: pass 1 groups equal keys by match_key, counts them
// per expert and overwrites s_key[i] with (key, group size, rank in group)
// packed in 22 bits (E <= 2048); pass 2 places from that record.  s_wc and the
// key groups [nw][E] that follow it in shared memory are zero on entry (the
// key groups are left zero).  The order never depends on timing.  Every
// thread of the block calls it (block barriers inside).
constexpr int kRankWarps = 8;
// Rank warps of the tiled path: 4 above 1024 experts, so that its counters and
// key groups (2 x warps x E ints) fit beside the staged entries.
__host__ __device__ inline int tiled_rank_warps(int E) { return E > 1024 ? kRankWarps / 2 : kRankWarps; }
__device__ void rank_entries(int* s_key, int n_ent, int E, const int* s_eb, int* s_wc, int32_t* out, int nw,
                             int64_t out_n, int32_t* status) {
    uint32_t* s_kb = reinterpret_cast<uint32_t*>(s_wc + nw * E);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunks = (n_ent + 31) / 32;
    const int per = (chunks + nw - 1) / nw;
    const int c0 = warp < nw ? min(chunks, warp * per) : 0;
    const int c1 = warp < nw ? min(chunks, c0 + per) : 0;
    for (int c = c0; c < c1; ++c) {                     // pass 1: per-(warp, expert) counts
        const int i = c * 32 + lane;
        const int key = i < n_ent ? s_key[i] : -1 - lane;
        const unsigned g = match_key(key, s_kb + warp * E, lane);
        if (key >= 0 && lane == __ffs(g) - 1) s_wc[warp * E + key] += __popc(g);
        if (key >= 0 && i < n_ent) s_key[i] = (key << 11) | (__popc(g) << 5) | __popc(g & ((1u << lane) - 1u));
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {   // per-warp bases, warps in entry order
        int run = s_eb[e];
        for (int w = 0; w < nw; ++w) {
            const int v = s_wc[w * E + e];
            s_wc[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    for (int c = c0; c < c1; ++c) {                     // pass 2: place
        const int i = c * 32 + lane;
        const int rec = i < n_ent ? s_key[i] : -1;   // key << 11 | group size << 5 | rank in group
        const int key = rec >> 11;
        int pos = -1;
        if (rec >= 0) pos = s_wc[warp * E + key] + (rec & 31);
        __syncwarp();
        if (rec >= 0 && (rec & 31) == 0) s_wc[warp * E + key] += (rec >> 5) & 63;
        __syncwarp();
        if (i < n_ent && ::epg::in_bounds(i, out_n, status)) out[i] = pos;
    }
}

// Expanded (per-expert) rows of one tile's (token, k) entries: expert e's
// entries take rows s_eb[e] (expert_offset[e] + entries of e in earlier
// tiles) + their stable rank in the tile, in (token, k) order.  The tile's
// entries are staged in shared memory (the first batch was loaded at kernel
// entry).  Needs 256 K + 2 x tiled_rank_warps(E) x E shared ints.
__device__ void expanded_rows_of_tile(const LayoutParams& p, int t0, int nt, const int* s_eb, int* sm,
                                      const int64_t (&key0)[kStageUnroll]) {
    const int E = p.E;
    const int n_ent = nt * p.K;
    int* s_key = sm;                        // [256 K] expert of each entry, or a unique negative
    const int nw = tiled_rank_warps(E);
    int* s_wc = s_key + kTileTokens * p.K;  // [nw][E] per-warp counts, then per-warp bases
    uint32_t* s_kb = reinterpret_cast<uint32_t*>(s_wc + nw * E);   // [nw][E] key groups
    const int64_t* src = p.topk_idx + static_cast<int64_t>(t0) * p.K;
    for (int base = 0; base < n_ent; base += kStageUnroll * kThreads) {
        int64_t e[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {   // the first batch was loaded at kernel entry
            const int i = base + u * kThreads + threadIdx.x;
            e[u] = base == 0 ? key0[u]
                             : ((i < n_ent && EP_IN(static_cast<int64_t>(t0) * p.K + i, static_cast<int64_t>(p.T) * p.K)) ? src[i] : -1);
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int i = base + u * kThreads + threadIdx.x;
            if (i < n_ent) s_key[i] = (e[u] >= 0 && e[u] < E) ? static_cast<int>(e[u]) : -1 - (i & 31);
        }
    }
    for (int i = threadIdx.x; i < nw * E; i += kThreads) {
        s_wc[i] = 0;
        s_kb[i] = 0u;
    }
    __syncthreads();
    rank_entries(s_key, n_ent, E, s_eb, s_wc, p.expanded_row + static_cast<int64_t>(t0) * p.K, nw,
                 static_cast<int64_t>(p.T - t0) * p.K, p.status);
}

// Node rows of one tile: a token is in node n when any rank of n holds it,
// so node n's membership word is the OR of its ranks' words; node n's rows
// are s_nbase[n] (node_offset[n] + its tokens in earlier tiles) + popc below
// the token.  Needs 2 * kTileWords * num_nodes shared ints; ends with a block
// barrier so the caller may reuse them.
__device__ void node_rows_of_tile(const LayoutParams& p, int t0, int nt, const uint32_t* s_bm, const int* s_nbase,
                                  int* sm) {
    const int NN = p.num_nodes, R = p.R, rpn = p.ranks_per_node;
    uint32_t* s_nbm = reinterpret_cast<uint32_t*>(sm);                // [kTileWords][NN]
    int* s_nwpre = reinterpret_cast<int*>(s_nbm + NN * kTileWords);    // [kTileWords][NN]
    for (int i = threadIdx.x; i < NN * kTileWords; i += kThreads) {
        const int w = i / NN;
        const int n = i - w * NN;
        uint32_t word = 0u;
        for (int r = n * rpn; r < (n + 1) * rpn; ++r) word |= s_bm[w * R + r];
        s_nbm[i] = word;
    }
    __syncthreads();
    for (int n = threadIdx.x; n < NN; n += kThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kTileWords; ++w) {
            s_nwpre[w * NN + n] = run;
            run += __popc(s_nbm[w * NN + n]);
        }
    }
    __syncthreads();
    int32_t* out = p.node_row + static_cast<size_t>(t0) * NN;
    for (int j = threadIdx.x; j < nt * NN; j += kThreads) {
        const int tl = j / NN;
        const int n = j - tl * NN;
        const int w = tl >> 5;
        const uint32_t word = s_nbm[w * NN + n];
        const uint32_t b = static_cast<uint32_t>(tl & 31);
        if (!EP_IN(static_cast<int64_t>(t0) * NN + j, static_cast<int64_t>(p.T) * NN)) continue;
        out[j] = ((word >> b) & 1u) ? s_nbase[n] + s_nwpre[w * NN + n] + __popc(word & ((1u << b) - 1u)) : -1;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) layout_rows_kernel(const LayoutParams p) {
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ int s_warp[kThreads / 32];
    const int R = p.R, E = p.E, NN = p.num_nodes;
    const int tile = blockIdx.x;
    const bool has_tile = tile < p.num_tiles;
    const bool expanded = p.expanded_row != nullptr && has_tile;
    const bool nodes = p.node_row != nullptr;
    int* s_base = reinterpret_cast<int*>(smem);                    // [R+1]
    uint32_t* s_bm = smem + (R + 1);                                // [kTileWords][R]
    int* s_wpre = reinterpret_cast<int*>(s_bm + R * kTileWords);    // [kTileWords][R]
    int* s_eb = s_wpre + R * kTileWords;                            // [E] expanded: expert bases
    int* s_nbase = s_eb + (p.expanded_row ? E : 0);                 // [NN] node bases
    int* s_extra = s_nbase + (nodes ? NN : 0);                      // node rows, then expanded rows
    pdl_wait();
    pdl_launch_dependents();   // the next kernel may be scheduled; it waits for our completion

    // Every independent global value this CTA needs, loaded at once (one
    // round trip): rank totals and this tile's rank prefixes, expert totals
    // (block 0: expert_offset; expanded: the ranking's bases) and this tile's
    // expert prefixes, node totals and prefixes, the tile's first top-k
    // entries, then its membership bitmaps.
    const int per_r = (R + kThreads - 1) / kThreads;
    const int per_e = (E + kThreads - 1) / kThreads;
    const int per_n = (NN + kThreads - 1) / kThreads;
    const bool want_e = tile == 0 || expanded;
    const bool want_n = nodes && (tile == 0 || has_tile);
    int v_cnt[kMaxRankSlice], v_wsr[kMaxRankSlice];
    int v_ce[kMaxExpertSlice], v_wse[kMaxExpertSlice];
    int v_cn[kMaxRankSlice], v_wsn[kMaxRankSlice];
    load_slice(v_cnt, R, per_r, true, [&](int i) { return p.num_tokens_per_rank[i]; });
    load_slice(v_wsr, R, per_r, has_tile, [&](int i) { return p.ws_rank[static_cast<size_t>(i) * p.num_tiles + tile]; });
    load_slice(v_ce, E, per_e, want_e, [&](int i) { return p.num_tokens_per_expert[i]; });
    load_slice(v_wse, E, per_e, expanded,
               [&](int i) { return p.ws_expert[static_cast<size_t>(i) * p.num_tiles + tile]; });
    load_slice(v_cn, NN, per_n, want_n, [&](int i) { return p.num_tokens_per_node[i]; });
    load_slice(v_wsn, NN, per_n, nodes && has_tile,
               [&](int i) { return p.ws_node[static_cast<size_t>(i) * p.num_tiles + tile]; });
    const int t0 = tile * kTileTokens;
    const int nt = has_tile ? min(kTileTokens, p.T - t0) : 0;
    int64_t key0[kStageUnroll];
    {
        const int n_ent = nt * p.K;
        const int64_t* src = p.topk_idx + static_cast<int64_t>(t0) * p.K;
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int i = u * kThreads + static_cast<int>(threadIdx.x);
            key0[u] = (expanded && i < n_ent && EP_IN(static_cast<int64_t>(t0) * p.K + i, static_cast<int64_t>(p.T) * p.K))
                          ? src[i] : -1;
        }
    }
    if (has_tile) {
        const uint32_t* g_bm = p.ws_bitmap + static_cast<size_t>(tile) * R * kTileWords;
        for (int base = 0; base < R * kTileWords; base += kStageUnroll * kThreads) {
            uint32_t v[kStageUnroll];
#pragma unroll
            for (int u = 0; u < kStageUnroll; ++u) {   // all loads in flight before any use
                const int i = base + u * kThreads + threadIdx.x;
                v[u] = (i < R * kTileWords && EP_IN(static_cast<int64_t>(tile) * R * kTileWords + i,
                                                    static_cast<int64_t>(p.num_tiles) * R * kTileWords))
                           ? g_bm[i] : 0u;
            }
#pragma unroll
            for (int u = 0; u < kStageUnroll; ++u) {
                const int i = base + u * kThreads + threadIdx.x;
                if (i < R * kTileWords) s_bm[i] = v[u];
            }
        }
    }

    // rank offsets, then this tile's base per rank
    {
        int pre[kMaxRankSlice];
        const int n_recv = block_exclusive_scan_slice(v_cnt, pre, per_r, s_warp);
#pragma unroll
        for (int j = 0; j < kMaxRankSlice; ++j) {
            const int i = static_cast<int>(threadIdx.x) * per_r + j;
            if (j < per_r && i < R) {
                if (tile == 0 && EP_IN(i, R + 1)) p.rank_offset[i] = pre[j];
                s_base[i] = pre[j] + v_wsr[j];
            }
        }
        if (tile == 0 && threadIdx.x == 0 && EP_IN(R, R + 1)) p.rank_offset[R] = n_recv;
    }
    // expert offsets (aligned counts): block 0 writes them; the expanded
    // ranking starts each expert at its offset plus this tile's prefix
    if (want_e) {
        const int a = p.alignment;
        int al[kMaxExpertSlice], pre[kMaxExpertSlice];
#pragma unroll
        for (int j = 0; j < kMaxExpertSlice; ++j) al[j] = (v_ce[j] + a - 1) / a * a;
        const int n_exp = block_exclusive_scan_slice(al, pre, per_e, s_warp);
#pragma unroll
        for (int j = 0; j < kMaxExpertSlice; ++j) {
            const int i = static_cast<int>(threadIdx.x) * per_e + j;
            if (j < per_e && i < E) {
                if (tile == 0 && EP_IN(i, E + 1)) p.expert_offset[i] = pre[j];
                if (expanded) s_eb[i] = pre[j] + v_wse[j];
            }
        }
        if (tile == 0 && threadIdx.x == 0 && EP_IN(E, E + 1)) p.expert_offset[E] = n_exp;
    }
    // node offsets and this tile's base per node
    if (want_n) {
        int pre[kMaxRankSlice];
        const int n_node = block_exclusive_scan_slice(v_cn, pre, per_n, s_warp);
#pragma unroll
        for (int j = 0; j < kMaxRankSlice; ++j) {
            const int i = static_cast<int>(threadIdx.x) * per_n + j;
            if (j < per_n && i < NN) {
                if (tile == 0 && EP_IN(i, NN + 1)) p.node_offset[i] = pre[j];
                s_nbase[i] = pre[j] + v_wsn[j];
            }
        }
        if (tile == 0 && threadIdx.x == 0 && EP_IN(NN, NN + 1)) p.node_offset[NN] = n_node;
    }
    if (!has_tile) {
        if (p.token_offset && p.num_tiles == 0 && threadIdx.x == 0) p.token_offset[0] = 0;
        return;
    }
    __syncthreads();   // s_base, s_bm (and the bases) visible
    for (int r = threadIdx.x; r < R; r += kThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kTileWords; ++w) {
            s_wpre[w * R + r] = run;
            run += __popc(s_bm[w * R + r]);
        }
    }
    __syncthreads();

    // dst_row and is_token_in_rank of the tile's contiguous [nt, R] block,
    // four entries per thread-step (16-byte / 4-byte stores)
    const int n_el = nt * R;
    int32_t* drow = p.dst_row + static_cast<size_t>(t0) * R;
    uint8_t* inr = p.is_token_in_rank + static_cast<size_t>(t0) * R;
    for (int q = threadIdx.x; q * 4 < n_el; q += kThreads) {
        const int j0 = q * 4;
        int tl = j0 / R;
        int r = j0 - tl * R;
        int v[4];
        uint32_t in4 = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            v[u] = -1;
            if (j0 + u < n_el) {
                const int w = tl >> 5;
                const uint32_t word = s_bm[w * R + r];
                const uint32_t b = static_cast<uint32_t>(tl & 31);
                if ((word >> b) & 1u) {
                    v[u] = s_base[r] + s_wpre[w * R + r] + __popc(word & ((1u << b) - 1u));
                    in4 |= 1u << (8 * u);
                }
            }
            if (++r == R) {
                r = 0;
                ++tl;
            }
        }
        if (j0 + 4 <= n_el) {
            if (EP_IN(static_cast<int64_t>(t0) * R + j0 + 3, static_cast<int64_t>(p.T) * R)) {
                *reinterpret_cast<int4*>(drow + j0) = make_int4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<uint32_t*>(inr + j0) = in4;
            }
        } else {
            for (int u = 0; u < 4 && j0 + u < n_el; ++u) {
                if (!EP_IN(static_cast<int64_t>(t0) * R + j0 + u, static_cast<int64_t>(p.T) * R)) continue;
                drow[j0 + u] = v[u];
                inr[j0 + u] = static_cast<uint8_t>((in4 >> (8 * u)) & 1u);
            }
        }
    }

    // token_offset: rows numbered token by token.  The rows of tokens before
    // this tile are the sum over ranks of the tile prefix of each rank.
    if (p.token_offset) {
        __shared__ int s_red[33];
        __shared__ int s_ntok[kTileTokens];
        int before = 0;
        for (int r = threadIdx.x; r < R; r += kThreads)
            if (EP_IN(static_cast<int64_t>(r) * p.num_tiles + tile, static_cast<int64_t>(R) * p.num_tiles))
                before += p.ws_rank[static_cast<size_t>(r) * p.num_tiles + tile];
        const int tile_base = block_sum(before, s_red);
        if (threadIdx.x < nt) {
            const int w = threadIdx.x >> 5;
            const uint32_t b = threadIdx.x & 31;
            int n = 0;
            for (int r = 0; r < R; ++r) n += (s_bm[w * R + r] >> b) & 1u;
            s_ntok[threadIdx.x] = n;
        }
        __syncthreads();
        const bool last = tile == p.num_tiles - 1;
        int32_t* to = p.token_offset + t0;
        block_exclusive_scan(
            nt, [&](int i) { return s_ntok[i]; },
            [&](int i, int v) {
                if ((i < nt || last) && EP_IN(t0 + i, p.T + 1)) to[i] = tile_base + v;
            },
            s_warp);
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
                c += __popc(s_bm[w * R + r] & mask);
            }
            if (c && EP_IN(s * R + r, R * R)) atomicAdd(&p.src_dst_count[s * R + r], c);
        }
    }

    if (nodes) node_rows_of_tile(p, t0, nt, s_bm, s_nbase, s_extra);
    if (expanded) expanded_rows_of_tile(p, t0, nt, s_eb, s_extra, key0);
}

// ---------------------------------------------------------------------------
// Single-launch cluster path
// ---------------------------------------------------------------------------

constexpr int kClusterThreads = 1024;
constexpr int kClusterUnroll = 4;
constexpr int kMaxClusterCtas = 16;
#ifndef EP_LAYOUT_CLUSTER_MAX_TOKEN_RANKS
#define EP_LAYOUT_CLUSTER_MAX_TOKEN_RANKS (1 << 19)
#endif
// Above this many (token, rank) outputs the tiled path (one CTA per 256 tokens) is used.
constexpr int64_t kClusterMaxTokenRanks = EP_LAYOUT_CLUSTER_MAX_TOKEN_RANKS;

// Shared-memory words of one cluster CTA for W bitmap words per rank.
// Warps that rank the expanded entries in a cluster CTA: all 32 while their
// [warps][E] counters stay small, else 8.
__host__ __device__ inline int cluster_rank_warps(int E) { return E <= 512 ? 32 : kRankWarps; }

size_t cluster_smem_words(int R, int E, int nodes, int W, int K, bool expanded, bool node_rows) {
    size_t w = 2 * static_cast<size_t>(R) * W + static_cast<size_t>(nodes) * W + R + E + nodes + (R + 1) + R +
               33 * static_cast<size_t>(W) + 64;
    if (expanded) w += 32 * static_cast<size_t>(W) * K + (1 + 2 * cluster_rank_warps(E)) * static_cast<size_t>(E);
    if (node_rows) w += 2 * static_cast<size_t>(nodes) + 1 + static_cast<size_t>(W) * nodes;
    return w;
}

// In-place exclusive scan of a[0, n) in shared memory by all kClusterThreads
// threads; returns the total.  s_warp holds 33 ints.
__device__ int smem_exclusive_scan(int* a, int n, int* s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kClusterThreads - 1) / kClusterThreads;
    const int begin = min(n, tid * per);
    const int end = min(n, begin + per);
    int local = 0;
    for (int i = begin; i < end; ++i) local += a[i];
    const int incl = warp_inclusive_scan(local);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = s_warp[lane];
        const int inc = warp_inclusive_scan(v);
        s_warp[lane] = inc - v;
        if (lane == 31) s_warp[32] = inc;
    }
    __syncthreads();
    int run = s_warp[warp] + incl - local;
    for (int i = begin; i < end; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    const int total = s_warp[32];
    __syncthreads();
    return total;
}

// Exclusive scan of a[0, n) in shared memory by one warp (each lane a
// contiguous run of at most kWarpScanMax / 32 values); returns the total.
constexpr int kWarpScanMax = 256;
__device__ int warp_exclusive_scan_smem(int* a, int n) {
    const int lane = threadIdx.x & 31;
    const int per = (n + 31) / 32;
    const int begin = min(n, lane * per);
    const int end = min(n, begin + per);
    int local = 0;
    for (int i = begin; i < end; ++i) local += a[i];
    const int incl = warp_inclusive_scan(local);
    int run = incl - local;
    for (int i = begin; i < end; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    return __shfl_sync(0xffffffffu, incl, 31);
}

// kExpanded: also the expanded per-expert rows; kNodeRows: also the node rows
// of the hierarchical path (separate instantiations, so the plain layout
// carries none of that work).
template <bool kExpanded, bool kNodeRows>
__global__ void __launch_bounds__(kClusterThreads, 1)
    layout_cluster_kernel(const LayoutParams p, int tokens_per_cta) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int me = static_cast<int>(cluster.block_rank());
    extern __shared__ __align__(16) uint32_t smem[];
    __shared__ int s_warp[33];
    __shared__ int s_bad;
    const int R = p.R, E = p.E, NN = p.num_nodes;
    const int W = tokens_per_cta / 32;
    uint32_t* s_bm = smem;                                          // [W][R] membership
    int* s_wbase = reinterpret_cast<int*>(s_bm + R * W);            // [W][R] row base per word
    uint32_t* s_bmn = reinterpret_cast<uint32_t*>(s_wbase + R * W);  // [W][NN] node membership
    int* s_cnt = reinterpret_cast<int*>(s_bmn + NN * W);            // [R]  read by every CTA
    int* s_hist = s_cnt + R;                                        // [E]  read by the last CTA
    int* s_ncnt = s_hist + E;                                       // [NN] read by the last CTA
    int* s_tot = s_ncnt + NN;                                       // [R+1]
    int* s_before = s_tot + R + 1;                                  // [R]
    int* s_ntok = s_before + R;                                     // [32 W] token's row within its word
    int* s_wtok = s_ntok + 32 * W;                                  // [W] rows of earlier words
    constexpr bool expanded = kExpanded;
    int* s_key = s_wtok + W;                                        // expanded: [32 W K] expert of each entry
    int* s_eb = s_key + (expanded ? 32 * W * p.K : 0);              // expanded: [E] expert bases
    int* s_wc = s_eb + (expanded ? E : 0);                          // expanded: [8][E] ranking counters
    uint32_t* s_kb = reinterpret_cast<uint32_t*>(s_wc + (expanded ? cluster_rank_warps(E) * E : 0));   // expanded: [nw][E] key groups
    int* s_ntot = reinterpret_cast<int*>(s_kb) + (expanded ? cluster_rank_warps(E) * E : 0);  // node rows: [NN+1] totals -> node_offset
    int* s_nbefore = s_ntot + (kNodeRows ? NN + 1 : 0);             // node rows: [NN] tokens of earlier CTAs
    int* s_nwbase = s_nbefore + (kNodeRows ? NN : 0);               // node rows: [W][NN] earlier words
    __shared__ int s_rows_total;                                    // read by later CTAs
    __shared__ int s_cta_base;
    __shared__ int s_totals[3];                                     // N, expert rows, node rows
    const int tid = threadIdx.x;
    const int t0 = me * tokens_per_cta;
    const int nt = max(0, min(tokens_per_cta, p.T - t0));
    pdl_wait();
    pdl_launch_dependents();   // the next kernel may be scheduled; it waits for our completion

    for (int i = tid; i < R * W; i += kClusterThreads) s_bm[i] = 0u;
    for (int i = tid; i < NN * W; i += kClusterThreads) s_bmn[i] = 0u;
    for (int i = tid; i < E; i += kClusterThreads) s_hist[i] = 0;
    if (tid == 0) s_bad = 0;
    if (p.src_dst_count) {
        for (int i = me * kClusterThreads + tid; i < R * R; i += C * kClusterThreads)
            if (EP_IN(i, R * R)) p.src_dst_count[i] = 0;
    }
    __syncthreads();

    // Phase 1: membership bitmaps and the expert histogram of this CTA's range.
    const int n_ent = nt * p.K;
    const int64_t* src = p.topk_idx + static_cast<int64_t>(t0) * p.K;
    bool bad = false;
    for (int base = 0; base < n_ent; base += kClusterUnroll * kClusterThreads) {
        int64_t e[kClusterUnroll];
#pragma unroll
        for (int u = 0; u < kClusterUnroll; ++u) {
            const int i = base + u * kClusterThreads + tid;
            e[u] = (i < n_ent && EP_IN(static_cast<int64_t>(t0) * p.K + i, static_cast<int64_t>(p.T) * p.K)) ? src[i] : -1;
        }
        if (expanded) {
#pragma unroll
            for (int u = 0; u < kClusterUnroll; ++u) {
                const int i = base + u * kClusterThreads + tid;
                if (i < n_ent) s_key[i] = (e[u] >= 0 && e[u] < E) ? static_cast<int>(e[u]) : -1 - (i & 31);
            }
        }
#pragma unroll
        for (int u = 0; u < kClusterUnroll; ++u) {
            if (e[u] == -1) continue;
            if (e[u] < -1 || e[u] >= E) { bad = true; continue; }
            const int i = base + u * kClusterThreads + tid;
            const int tl = i / p.K;
            const int r = static_cast<int>(e[u]) / p.experts_per_rank;
            const uint32_t bit = 1u << (tl & 31);
            atomicAdd(&s_hist[e[u]], 1);
            atomicOr(&s_bm[(tl >> 5) * R + r], bit);
            if (NN) atomicOr(&s_bmn[(tl >> 5) * NN + r / p.ranks_per_node], bit);
        }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    for (int r = tid; r < R; r += kClusterThreads) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            s_wbase[w * R + r] = run;
            run += __popc(s_bm[w * R + r]);
        }
        s_cnt[r] = run;
    }
    for (int n = tid; n < NN; n += kClusterThreads) {
        int c = 0;
        for (int w = 0; w < W; ++w) {
            if (kNodeRows) s_nwbase[w * NN + n] = c;
            c += __popc(s_bmn[w * NN + n]);
        }
        s_ncnt[n] = c;
    }
    // Rows numbered token by token: one warp per 32-token word, lane = token.
    const int warp_id = tid >> 5, lane = tid & 31;
    for (int w = warp_id; w < W; w += kClusterThreads / 32) {
        int n = 0;
        for (int r = 0; r < R; ++r) n += (s_bm[w * R + r] >> lane) & 1u;
        const int incl = warp_inclusive_scan(n);
        s_ntok[w * 32 + lane] = incl - n;
        if (lane == 31) s_wtok[w] = incl;
    }
    if (tid == 0 && s_bad) atomicOr(p.status, EP_ERR_INVALID_INDEX);
    __syncthreads();
    if (warp_id == 0) {
        int carry = 0;
        for (int base = 0; base < W; base += 32) {
            const int v = base + lane < W ? s_wtok[base + lane] : 0;
            const int incl = warp_inclusive_scan(v);
            if (base + lane < W) s_wtok[base + lane] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_rows_total = carry;
    }
    cluster.sync();   // counts of every CTA visible; src_dst_count zeroed

    // Phase 2: rank totals and this CTA's base per rank (every CTA), expert and
    // node totals (the last CTA), all from the other CTAs' shared memory.
    // Remote loads are issued for all CTAs before any is summed (one latency).
    for (int r = tid; r < R; r += kClusterThreads) {
        int v[kMaxClusterCtas];
#pragma unroll
        for (int c = 0; c < kMaxClusterCtas; ++c) v[c] = c < C ? cluster.map_shared_rank(s_cnt, c)[r] : 0;
        int tot = 0, before = 0;
#pragma unroll
        for (int c = 0; c < kMaxClusterCtas; ++c) {
            tot += v[c];
            if (c < me) before += v[c];
        }
        s_tot[r] = tot;
        s_before[r] = before;
        if (me == 0 && EP_IN(r, R)) p.num_tokens_per_rank[r] = tot;
    }
    if (warp_id == 1) {
        const int v = lane < me ? *cluster.map_shared_rank(&s_rows_total, lane) : 0;
        const int sum = warp_inclusive_scan(v);
        if (lane == 31) s_cta_base = sum;
    }
    if (expanded) {
        // every CTA needs each expert's total (for the offsets) and its count in
        // earlier CTAs; the histograms stay untouched (others read them too)
        for (int e = tid; e < E; e += kClusterThreads) {
            int v[kMaxClusterCtas];
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) v[c] = c < C ? cluster.map_shared_rank(s_hist, c)[e] : 0;
            int tot = 0, before = 0;
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) {
                tot += v[c];
                if (c < me) before += v[c];
            }
            if (me == C - 1 && EP_IN(e, E)) p.num_tokens_per_expert[e] = tot;
            s_eb[e] = (tot + p.alignment - 1) / p.alignment * p.alignment;
            s_wc[e] = before;
        }
    }
    if (me == C - 1) {
        // only this CTA reads any s_hist, and each e is read and rewritten by one thread
        for (int e = tid; e < E && !expanded; e += kClusterThreads) {
            int v[kMaxClusterCtas];
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) v[c] = c < C ? cluster.map_shared_rank(s_hist, c)[e] : 0;
            int tot = 0;
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) tot += v[c];
            if (EP_IN(e, E)) p.num_tokens_per_expert[e] = tot;
            s_hist[e] = (tot + p.alignment - 1) / p.alignment * p.alignment;
        }
        for (int n = tid; n < NN && !kNodeRows; n += kClusterThreads) {
            int v[kMaxClusterCtas];
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) v[c] = c < C ? cluster.map_shared_rank(s_ncnt, c)[n] : 0;
            int tot = 0;
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) tot += v[c];
            if (EP_IN(n, NN)) p.num_tokens_per_node[n] = tot;
        }
    }
    if (kNodeRows) {
        // every CTA needs each node's total (for node_offset) and its tokens in
        // earlier CTAs
        for (int n = tid; n < NN; n += kClusterThreads) {
            int v[kMaxClusterCtas];
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) v[c] = c < C ? cluster.map_shared_rank(s_ncnt, c)[n] : 0;
            int tot = 0, before = 0;
#pragma unroll
            for (int c = 0; c < kMaxClusterCtas; ++c) {
                tot += v[c];
                if (c < me) before += v[c];
            }
            if (me == C - 1 && EP_IN(n, NN)) p.num_tokens_per_node[n] = tot;
            s_ntot[n] = tot;
            s_nbefore[n] = before;
        }
    }
    __syncthreads();
    // Exclusive scans: s_tot becomes rank_offset (every CTA), s_hist
    // expert_offset (last CTA); one warp each when short, else the block.
    if (R <= kWarpScanMax) {
        if (warp_id == 0) {
            const int tot = warp_exclusive_scan_smem(s_tot, R);
            if (lane == 0) s_totals[0] = tot;
        }
    } else {
        const int tot = smem_exclusive_scan(s_tot, R, s_warp);
        if (tid == 0) s_totals[0] = tot;
    }
    int* s_escan = expanded ? s_eb : s_hist;   // aligned expert totals -> expert_offset
    if (expanded || me == C - 1) {
        if (E <= kWarpScanMax) {
            if (warp_id == 2) {
                const int tot = warp_exclusive_scan_smem(s_escan, E);
                if (lane == 0) s_totals[1] = tot;
            }
        } else {
            const int tot = smem_exclusive_scan(s_escan, E, s_warp);
            if (tid == 0) s_totals[1] = tot;
        }
    }
    if (kNodeRows) {   // s_ntot becomes node_offset
        if (NN <= kWarpScanMax) {
            if (warp_id == 4) {
                const int tot = warp_exclusive_scan_smem(s_ntot, NN);
                if (lane == 0) s_totals[2] = tot;
            }
        } else {
            const int tot = smem_exclusive_scan(s_ntot, NN, s_warp);
            if (tid == 0) s_totals[2] = tot;
        }
    }
    __syncthreads();
    const int n_recv = s_totals[0];
    if (me == 0) {
        for (int r = tid; r < R; r += kClusterThreads)
            if (EP_IN(r, R + 1)) p.rank_offset[r] = s_tot[r];
        if (tid == 0 && EP_IN(R, R + 1)) p.rank_offset[R] = n_recv;
    }
    if (me == C - 1) {
        for (int e = tid; e < E; e += kClusterThreads)
            if (EP_IN(e, E + 1)) p.expert_offset[e] = s_escan[e];
        if (tid == 0 && EP_IN(E, E + 1)) p.expert_offset[E] = s_totals[1];
        if (kNodeRows) {
            for (int n = tid; n < NN; n += kClusterThreads)
                if (EP_IN(n, NN + 1)) p.node_offset[n] = s_ntot[n];
            if (tid == 0 && EP_IN(NN, NN + 1)) p.node_offset[NN] = s_totals[2];
        }
    }

    // Phase 3: dst_row and is_token_in_rank of this CTA's [nt, R] block:
    // rank_offset + rows of earlier CTAs + rows of earlier words + popc below.
    const int n_el = nt * R;
    int32_t* drow = p.dst_row + static_cast<int64_t>(t0) * R;
    uint8_t* inr = p.is_token_in_rank + static_cast<int64_t>(t0) * R;
    for (int q = tid; q * 4 < n_el; q += kClusterThreads) {
        const int j0 = q * 4;
        int tl = j0 / R;
        int r = j0 - tl * R;
        int v[4];
        uint32_t in4 = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            v[u] = -1;
            if (j0 + u < n_el) {
                const int w = tl >> 5;
                const uint32_t word = s_bm[w * R + r];
                const uint32_t b = static_cast<uint32_t>(tl & 31);
                if ((word >> b) & 1u) {
                    v[u] = s_tot[r] + s_before[r] + s_wbase[w * R + r] + __popc(word & ((1u << b) - 1u));
                    in4 |= 1u << (8 * u);
                }
            }
            if (++r == R) { r = 0; ++tl; }
        }
        if (j0 + 4 <= n_el) {
            if (EP_IN(static_cast<int64_t>(t0) * R + j0 + 3, static_cast<int64_t>(p.T) * R)) {
                *reinterpret_cast<int4*>(drow + j0) = make_int4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<uint32_t*>(inr + j0) = in4;
            }
        } else {
            for (int u = 0; u < 4 && j0 + u < n_el; ++u) {
                if (!EP_IN(static_cast<int64_t>(t0) * R + j0 + u, static_cast<int64_t>(p.T) * R)) continue;
                drow[j0 + u] = v[u];
                inr[j0 + u] = static_cast<uint8_t>((in4 >> (8 * u)) & 1u);
            }
        }
    }

    // Rows-ready signal: this CTA's dst_row block is complete.  The reader
    // count is cleared before the tag goes out (readers count only once
    // they have seen it), and the block's stores are ordered before the tag
    // by the barrier and the fence.
    if (p.rows_ready) {
        __syncthreads();
        if (tid == 0) {
            uint64_t* slot = p.rows_ready + static_cast<size_t>(me) * kReadyWords;
            *reinterpret_cast<volatile uint32_t*>(slot + 1) = 0u;
            __threadfence();
            st_release_u64(slot, p.rows_tag);
        }
    }

    // Node rows of this CTA's [nt, nodes] block: node_offset + tokens of
    // earlier CTAs + tokens of earlier words + popc below.
    if (kNodeRows) {
        int32_t* nrow = p.node_row + static_cast<int64_t>(t0) * NN;
        for (int j = tid; j < nt * NN; j += kClusterThreads) {
            const int tl = j / NN;
            const int n = j - tl * NN;
            const int w = tl >> 5;
            const uint32_t word = s_bmn[w * NN + n];
            const uint32_t b = static_cast<uint32_t>(tl & 31);
            if (!EP_IN(static_cast<int64_t>(t0) * NN + j, static_cast<int64_t>(p.T) * NN)) continue;
            nrow[j] = ((word >> b) & 1u)
                          ? s_ntot[n] + s_nbefore[n] + s_nwbase[w * NN + n] + __popc(word & ((1u << b) - 1u))
                          : -1;
        }
    }

    // token_offset: rows of earlier CTAs' tokens + rows of earlier words + row in word.
    if (p.token_offset) {
        const int cta_base = s_cta_base;
        for (int tl = tid; tl < nt; tl += kClusterThreads)
            if (EP_IN(t0 + tl, p.T + 1)) p.token_offset[t0 + tl] = cta_base + s_wtok[tl >> 5] + s_ntok[tl];
        if (me == C - 1 && tid == 0 && EP_IN(p.T, p.T + 1)) p.token_offset[p.T] = n_recv;
    }

    // src_dst_count[s][r] += tokens of source rank s in this range that rank r receives.
    if (p.src_dst_count && nt > 0) {
        const int ts = p.T / R;
        const int s_lo = t0 / ts;
        const int s_hi = (t0 + nt - 1) / ts;
        const int n_pairs = (s_hi - s_lo + 1) * R;
        for (int q = tid; q < n_pairs; q += kClusterThreads) {
            const int s = s_lo + q / R;
            const int r = q - (q / R) * R;
            const int a = max(t0, s * ts) - t0;
            const int b = min(t0 + nt, (s + 1) * ts) - t0;
            int c = 0;
            for (int w = a >> 5; w <= (b - 1) >> 5; ++w) {
                const int lo = max(a - w * 32, 0);
                const int hi = min(b - w * 32, 32);
                const uint32_t upper = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
                c += __popc(s_bm[w * R + r] & upper & ~((1u << lo) - 1u));
            }
            if (c && EP_IN(s * R + r, R * R)) atomicAdd(&p.src_dst_count[s * R + r], c);
        }
    }
    // Expanded rows: expert e's entries of this CTA start at expert_offset[e] +
    // its entries in earlier CTAs and are ranked in (token, k) order.
    if (expanded) {
        const int nw = cluster_rank_warps(E);
        for (int e = tid; e < E; e += kClusterThreads) {
            s_eb[e] += s_wc[e];   // each thread owns column e of s_wc here
            for (int w = 0; w < nw; ++w) {
                s_wc[w * E + e] = 0;
                s_kb[w * E + e] = 0u;
            }
        }
        __syncthreads();
        rank_entries(s_key, n_ent, E, s_eb, s_wc, p.expanded_row + static_cast<int64_t>(t0) * p.K, nw,
                     static_cast<int64_t>(p.T - t0) * p.K, p.status);
    }

    // No CTA may exit (releasing its shared memory) while another still reads it.
    cluster.sync();
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Cluster shape for the single-launch path, or C = 0 when it does not apply.
struct ClusterPlan {
    int ctas;
    int tokens_per_cta;
    size_t smem;
};

// Few tokens (T <= 1024, R <= 32, K <= 16, no node rows): one CTA of 1024
// threads and no cluster.  Every phase is spread over all 32 warps, whatever
// T: the top-k entries one per thread (shared atomics build the [word][rank]
// bitmaps and the expert histogram), one warp per rank for its prefix over
// words, one per word for its tokens' rows and one per 32 experts for their
// aligned counts, then (token, rank) quads of dst_row and is_token_in_rank
// per thread.  Three block barriers (a fourth and the ranking's two with
// expanded rows), no cluster barrier and no remote read.
#ifndef EP_LAYOUT_SMALL_MAX_TOKENS
#define EP_LAYOUT_SMALL_MAX_TOKENS 1024   // 0 disables the single-CTA path
#endif
constexpr int kSmallMaxTokens = EP_LAYOUT_SMALL_MAX_TOKENS <= 1024 ? EP_LAYOUT_SMALL_MAX_TOKENS : 1024;
constexpr int kSmallMaxRanks = 32;
constexpr int kSmallMaxTopk = 16;
constexpr int kSmallEntries = kSmallMaxTopk;   // entries per thread: <= 1024 tokens x 16 over 1024 threads
constexpr int kSmallRankWarps = 8;             // warps ranking the expanded entries

// Dynamic shared memory of the single-CTA kernel, in ints: the expert
// histogram, and with expanded rows the entries' experts and the ranking's
// per-(warp, expert) counters.
inline size_t small_smem_ints(int E, int n_ent, bool expanded) {
    return static_cast<size_t>(E) + (expanded ? static_cast<size_t>(n_ent) + 2 * static_cast<size_t>(kSmallRankWarps) * E : 0);
}

// kExpanded: also the expanded rows (each valid (t, k) numbered within its
// expert in (token, k) order from expert_offset), ranked after the offsets.
// kNodeRows: also node_offset and the node rows, formed like the rank rows
// from the [word][node] bitmaps.
template <bool kExpanded, bool kNodeRows>
__global__ void __launch_bounds__(1024, 1) layout_small_kernel(const LayoutParams p) {
    __shared__ uint32_t s_bm[32][kSmallMaxRanks + 1];    // [word][rank] membership
    __shared__ int s_base[32][kSmallMaxRanks + 1];       // [word][rank] rows in earlier words
    __shared__ uint32_t s_bmn[32][kSmallMaxRanks + 1];   // [word][node] membership
    __shared__ int s_nbase[kNodeRows ? 32 : 1][kSmallMaxRanks + 1];   // [word][node] tokens in earlier words
    __shared__ int s_ntot[kSmallMaxRanks];               // node rows: tokens of each node
    __shared__ int s_tot[kSmallMaxRanks];                // rows of each rank
    __shared__ int s_ntok[1024];                         // token's row within its word
    __shared__ int s_wtok[32];                           // rows of each word
    __shared__ int s_echunk[64];                         // aligned rows of each 32-expert chunk
    __shared__ int s_bad;
    extern __shared__ int s_hist[];                      // [E] entries per expert
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T, K = p.K, E = p.E, R = p.R, NN = p.num_nodes;
    const int W = (T + 31) >> 5;
    const int n_ent = T * K;
    int* s_key = s_hist + E;                              // expanded: [n_ent] expert of each entry
    int* s_wc = s_key + (kExpanded ? n_ent : 0);          // expanded: [8][E] ranking counters
    uint32_t* s_kb = reinterpret_cast<uint32_t*>(s_wc + (kExpanded ? kSmallRankWarps * E : 0));   // expanded: [8][E] key groups
    pdl_wait();
    pdl_launch_dependents();

    // this thread's top-k entries, in flight while shared memory is cleared
    int64_t v[kSmallEntries];
#pragma unroll
    for (int u = 0; u < kSmallEntries; ++u) {
        const int i = u * 1024 + tid;
        v[u] = i < n_ent ? p.topk_idx[i] : -1;
    }
    for (int i = tid; i < 32 * (kSmallMaxRanks + 1); i += 1024) {
        (&s_bm[0][0])[i] = 0u;
        (&s_bmn[0][0])[i] = 0u;
    }
    for (int i = tid; i < E; i += 1024) s_hist[i] = 0;
    if (kExpanded)
        for (int i = tid; i < kSmallRankWarps * E; i += 1024) {
            s_wc[i] = 0;
            s_kb[i] = 0u;
        }
    if (tid == 0) s_bad = 0;
    __syncthreads();

    // Phase 1: bitmaps and expert histogram.
    bool bad = false;
#pragma unroll
    for (int u = 0; u < kSmallEntries; ++u) {
        const int64_t e = v[u];
        if (kExpanded) {
            const int i = u * 1024 + tid;
            if (i < n_ent) s_key[i] = (e >= 0 && e < E) ? static_cast<int>(e) : -1 - (i & 31);
        }
        if (e == -1) continue;
        if (e < -1 || e >= E) {
            bad = true;
            continue;
        }
        const int tk = (u * 1024 + tid) / K;
        const int r = static_cast<int>(e) / p.experts_per_rank;
        const uint32_t bit = 1u << (tk & 31);
        atomicAdd(&s_hist[e], 1);
        atomicOr(&s_bm[tk >> 5][r], bit);
        if (NN) atomicOr(&s_bmn[tk >> 5][r / p.ranks_per_node], bit);
    }
    if (bad) s_bad = 1;
    __syncthreads();

    // Phase 2: warp r scans rank r over the words (and fills column r of
    // src_dst_count), warp n totals node n, warp w numbers word w's tokens,
    // and warp c scans the aligned counts of experts [32c, 32c + 32).
    if (warp < R) {
        const int r = warp;
        const int c = lane < W ? __popc(s_bm[lane][r]) : 0;
        const int incl = warp_inclusive_scan(c);
        if (lane < W) s_base[lane][r] = incl - c;
        if (lane == 31) {
            s_tot[r] = incl;
            p.num_tokens_per_rank[r] = incl;
        }
        if (p.src_dst_count && lane < R) {   // src_dst_count[s][r], s = lane (R | T)
            const int ts = T / R;
            const int a = lane * ts, b = a + ts;
            int cnt = 0;
            for (int w = a >> 5; w < W && w * 32 < b; ++w) {
                const int lo = max(a - w * 32, 0), hi = min(b - w * 32, 32);
                const uint32_t upper = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
                cnt += __popc(s_bm[w][r] & upper & ~((1u << lo) - 1u));
            }
            p.src_dst_count[lane * R + r] = cnt;
        }
    }
    if (warp < NN) {
        const int c = lane < W ? __popc(s_bmn[lane][warp]) : 0;
        if (kNodeRows) {   // warp n: node n's prefix over the words
            const int incl = warp_inclusive_scan(c);
            if (lane < W) s_nbase[lane][warp] = incl - c;
            if (lane == 31) {
                s_ntot[warp] = incl;
                p.num_tokens_per_node[warp] = incl;
            }
        } else {
            const int tot = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c)));
            if (lane == 0) p.num_tokens_per_node[warp] = tot;
        }
    }
    if (warp < W) {
        int n = 0;
        for (int r = 0; r < R; ++r) n += (s_bm[warp][r] >> lane) & 1u;
        const int incl = warp_inclusive_scan(n);
        s_ntok[warp * 32 + lane] = incl - n;
        if (lane == 31) s_wtok[warp] = incl;
    }
    const int n_chunks = (E + 31) >> 5;   // <= 64
    for (int c = warp; c < n_chunks; c += 32) {
        const int e = c * 32 + lane;
        const int cnt = e < E ? s_hist[e] : 0;
        if (e < E) p.num_tokens_per_expert[e] = cnt;
        const int al = (cnt + p.alignment - 1) / p.alignment * p.alignment;
        const int incl = warp_inclusive_scan(al);
        if (e < E) s_hist[e] = incl - al;   // exclusive within the chunk
        if (lane == 31) s_echunk[c] = incl;
    }
    __syncthreads();

    // Phase 3: every warp forms rank_offset (lane r) and the words' row bases
    // (lane w) by shuffles, then writes (token, rank) quads and token offsets.
    const int tv = lane < R ? s_tot[lane] : 0;
    const int tincl = warp_inclusive_scan(tv);
    const int ro = tincl - tv;
    const int n_recv = __shfl_sync(0xffffffffu, tincl, 31);
    const int wv = lane < W ? s_wtok[lane] : 0;
    const int wincl = warp_inclusive_scan(wv);
    const int wbase = wincl - wv;
    // expert offsets: chunk bases (chunks lane and 32 + lane) + row within the chunk
    if (warp < n_chunks) {
        const int c0 = lane < n_chunks ? s_echunk[lane] : 0;
        const int c1 = 32 + lane < n_chunks ? s_echunk[32 + lane] : 0;
        const int i0 = warp_inclusive_scan(c0);
        const int t0 = __shfl_sync(0xffffffffu, i0, 31);
        const int i1 = warp_inclusive_scan(c1);
        for (int c = warp; c < n_chunks; c += 32) {   // warp-uniform
            const int base = c < 32 ? __shfl_sync(0xffffffffu, i0 - c0, c)
                                    : t0 + __shfl_sync(0xffffffffu, i1 - c1, c - 32);
            const int e = c * 32 + lane;
            if (e < E) {
                p.expert_offset[e] = base + s_hist[e];
                if (kExpanded) s_hist[e] += base;   // now expert_offset, the ranking's bases
            }
        }
        const int t1 = __shfl_sync(0xffffffffu, i1, 31);
        if (warp == 0 && lane == 0) p.expert_offset[E] = t0 + t1;
    }
    if (warp == 0) {
        if (lane < R) p.rank_offset[lane] = ro;
        if (lane == 0) {
            p.rank_offset[R] = n_recv;
            if (p.token_offset) p.token_offset[T] = n_recv;
            if (s_bad) atomicOr(p.status, EP_ERR_INVALID_INDEX);
        }
    }
    if (p.token_offset) {
        for (int t0 = warp * 32; t0 < T; t0 += 1024) {   // warp-uniform
            const int base = __shfl_sync(0xffffffffu, wbase, (t0 >> 5) & 31);
            if (t0 + lane < T) p.token_offset[t0 + lane] = base + s_ntok[t0 + lane];
        }
    }
    const int n_el = T * R;
    // j / R as a multiply-high: m = ceil(2^32 / R) is exact for j < 2^27
    const uint32_t m_r = R > 1 ? 0xffffffffu / static_cast<uint32_t>(R) + 1u : 0u;
    for (int q0 = warp * 128; q0 < n_el; q0 += 4096) {   // warp-uniform; 4 outputs per lane
        const int j0 = q0 + lane * 4;
        int tl = R > 1 ? static_cast<int>(__umulhi(static_cast<uint32_t>(j0), m_r)) : j0;
        int r = j0 - tl * R;
        int d[4];
        uint32_t in4 = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int ror = __shfl_sync(0xffffffffu, ro, r & 31);
            d[u] = -1;
            if (j0 + u < n_el) {
                const int w = tl >> 5;
                const uint32_t word = s_bm[w][r];
                const uint32_t b = static_cast<uint32_t>(tl & 31);
                if ((word >> b) & 1u) {
                    d[u] = ror + s_base[w][r] + __popc(word & ((1u << b) - 1u));
                    in4 |= 1u << (8 * u);
                }
            }
            if (++r == R) {
                r = 0;
                ++tl;
            }
        }
        if (j0 + 4 <= n_el) {
            *reinterpret_cast<int4*>(p.dst_row + j0) = make_int4(d[0], d[1], d[2], d[3]);
            *reinterpret_cast<uint32_t*>(p.is_token_in_rank + j0) = in4;
        } else {
            for (int u = 0; u < 4 && j0 + u < n_el; ++u) {
                p.dst_row[j0 + u] = d[u];
                p.is_token_in_rank[j0 + u] = static_cast<uint8_t>((in4 >> (8 * u)) & 1u);
            }
        }
    }
    if (kNodeRows) {   // node_offset (lane n) by shuffles, then (token, node) quads
        const int nv = lane < NN ? s_ntot[lane] : 0;
        const int nincl = warp_inclusive_scan(nv);
        const int no = nincl - nv;
        if (warp == 0) {
            if (lane < NN) p.node_offset[lane] = no;
            const int n_node = __shfl_sync(0xffffffffu, nincl, 31);
            if (lane == 0) p.node_offset[NN] = n_node;
        }
        const int n_eln = T * NN;
        const uint32_t m_n = NN > 1 ? 0xffffffffu / static_cast<uint32_t>(NN) + 1u : 0u;
        for (int q0 = warp * 128; q0 < n_eln; q0 += 4096) {   // warp-uniform
            const int j0 = q0 + lane * 4;
            int tl = NN > 1 ? static_cast<int>(__umulhi(static_cast<uint32_t>(j0), m_n)) : j0;
            int n = j0 - tl * NN;
            int d[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int nor = __shfl_sync(0xffffffffu, no, n & 31);
                d[u] = -1;
                if (j0 + u < n_eln) {
                    const int w = tl >> 5;
                    const uint32_t word = s_bmn[w][n];
                    const uint32_t b = static_cast<uint32_t>(tl & 31);
                    if ((word >> b) & 1u) d[u] = nor + s_nbase[w][n] + __popc(word & ((1u << b) - 1u));
                }
                if (++n == NN) {
                    n = 0;
                    ++tl;
                }
            }
            if (j0 + 4 <= n_eln) {
                *reinterpret_cast<int4*>(p.node_row + j0) = make_int4(d[0], d[1], d[2], d[3]);
            } else {
                for (int u = 0; u < 4 && j0 + u < n_eln; ++u) p.node_row[j0 + u] = d[u];
            }
        }
    }
    if (kExpanded) {
        __syncthreads();   // s_hist now holds expert_offset
        rank_entries(s_key, n_ent, E, s_hist, s_wc, p.expanded_row, kSmallRankWarps,
                     static_cast<int64_t>(p.T) * p.K, p.status);
    }
}

// Largest static shared memory of the cluster kernel instantiations so far.
template <bool kX, bool kN>
cudaError_t cluster_static_smem(int& bytes) {
    cudaFuncAttributes fa{};
    const cudaError_t e = cudaFuncGetAttributes(&fa, layout_cluster_kernel<kX, kN>);
    if (e == cudaSuccess && static_cast<int>(fa.sharedSizeBytes) > bytes) bytes = static_cast<int>(fa.sharedSizeBytes);
    return e;
}

template <bool kX, bool kN>
bool configure_cluster(int smem_max) {
    return cudaFuncSetAttribute(layout_cluster_kernel<kX, kN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_max) == cudaSuccess &&
           cudaFuncSetAttribute(layout_cluster_kernel<kX, kN>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
               cudaSuccess;
}

ClusterPlan plan_cluster(const LayoutParams& p, int smem_max) {
    ClusterPlan plan{0, 0, 0};
    // One CTA per 256 tokens up to 16; ranges are whole 32-token words.
    int ctas = (p.T + kTileTokens - 1) / kTileTokens;
    if (ctas < 1) ctas = 1;
    if (ctas > kMaxClusterCtas) ctas = kMaxClusterCtas;
    int tpc = (p.T + ctas - 1) / ctas;
    tpc = (tpc + 31) / 32 * 32;
    if (tpc < 32) tpc = 32;
    ctas = (p.T + tpc - 1) / tpc;
    if (ctas < 1) ctas = 1;
    const size_t smem = 4 * cluster_smem_words(p.R, p.E, p.num_nodes, tpc / 32, p.K, p.expanded_row != nullptr,
                                               p.node_row != nullptr);
    if (smem > static_cast<size_t>(smem_max)) return plan;
    // Large [T, R] outputs are written faster by the many-CTA path.
    if (static_cast<int64_t>(p.T) * p.R > kClusterMaxTokenRanks) return plan;
    plan.ctas = ctas;
    plan.tokens_per_cta = tpc;
    plan.smem = smem;
    return plan;
}

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

cudaError_t launch_layout(const LayoutParams& p_in, cudaStream_t stream, RowsSignal* sig) {
    const DeviceInfo& di = device_info();
    LayoutParams p = p_in;
    p.rows_ready = nullptr;   // only the cluster kernel publishes, when sig has room for its lines
    p.rows_tag = 0;
    if (sig) {
        sig->tokens = 0;
        sig->count = 0;
    }
    static thread_local int configured_device = -1;
    static thread_local bool cluster_ok = false;
    static thread_local int cluster_smem_max = 0;
    if (configured_device != di.device) {
        // Worst case over the supported limits (R = 1024, E = 2048): < 80 KB.
        const int cap = di.max_smem_optin < 100 * 1024 ? di.max_smem_optin : 100 * 1024;
        cudaError_t e = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
        if (e != cudaSuccess) return e;
        // the rows kernel needs up to ~220 KB with expanded rows: all the dynamic
        // shared memory the block limit leaves beside its static shared memory
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, layout_rows_kernel);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(layout_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 di.max_smem_optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        int static_smem = 0;
        e = cluster_static_smem<false, false>(static_smem);
        if (e == cudaSuccess) e = cluster_static_smem<true, false>(static_smem);
        if (e == cudaSuccess) e = cluster_static_smem<false, true>(static_smem);
        if (e == cudaSuccess) e = cluster_static_smem<true, true>(static_smem);
        if (e != cudaSuccess) return e;
        cluster_smem_max = di.max_smem_optin - static_smem;
        // the single-CTA kernel with expanded rows: up to ~140 KB at the limits
        const int small_max = static_cast<int>(4 * small_smem_ints(EP_MAX_EXPERTS, kSmallMaxTokens * kSmallMaxTopk, true));
        e = cudaFuncSetAttribute(layout_small_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, small_max);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(layout_small_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, small_max);
        if (e != cudaSuccess) return e;
        cluster_ok = configure_cluster<false, false>(cluster_smem_max) &&
                     configure_cluster<true, false>(cluster_smem_max) &&
                     configure_cluster<false, true>(cluster_smem_max) && configure_cluster<true, true>(cluster_smem_max);
        cudaGetLastError();   // a refused attribute only disables the cluster path
        configured_device = di.device;
    }

    if (p.T <= kSmallMaxTokens && p.R <= kSmallMaxRanks && p.K <= kSmallMaxTopk) {
        const bool expanded = p.expanded_row != nullptr, nodes = p.node_row != nullptr;
        const size_t smem = 4 * small_smem_ints(p.E, p.T * p.K, expanded);
        auto kernel = expanded ? (nodes ? layout_small_kernel<true, true> : layout_small_kernel<true, false>)
                               : (nodes ? layout_small_kernel<false, true> : layout_small_kernel<false, false>);
        if (sig) sig->slots = nullptr;
        return launch_pdl(kernel, dim3(1), dim3(1024), smem, stream, p);
    }

    const ClusterPlan plan = cluster_ok ? plan_cluster(p, cluster_smem_max) : ClusterPlan{0, 0, 0};
    if (plan.ctas > 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = plan.ctas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(plan.ctas);
        cfg.blockDim = dim3(kClusterThreads);
        cfg.dynamicSmemBytes = plan.smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        int max_clusters = 0;
        cfg.numAttrs = 1;   // the occupancy query takes the cluster shape only
        const bool expanded = p.expanded_row != nullptr, nodes = p.node_row != nullptr;
        auto kernel = expanded ? (nodes ? layout_cluster_kernel<true, true> : layout_cluster_kernel<true, false>)
                               : (nodes ? layout_cluster_kernel<false, true> : layout_cluster_kernel<false, false>);
        const bool fits = cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &cfg) == cudaSuccess;
        cfg.numAttrs = 2;
        if (fits && max_clusters >= 1) {
            if (sig && sig->slots && static_cast<size_t>(plan.ctas) * kReadyWords * 8 <= sig->bytes) {
                p.rows_ready = sig->slots;
                p.rows_tag = sig->tag;
                sig->tokens = plan.tokens_per_cta;
                sig->count = plan.ctas;
            } else if (sig) {
                sig->slots = nullptr;
            }
            if (debug_enabled())
                debug_launch(reinterpret_cast<const void*>(kernel), cfg.gridDim, cfg.blockDim, plan.smem, plan.ctas);
            return cudaLaunchKernelEx(&cfg, kernel, p, plan.tokens_per_cta);
        }
        cudaGetLastError();   // fall back to the tiled path
    }
    if (sig) sig->slots = nullptr;

    const size_t smem_count =
        4 * (static_cast<size_t>(p.R) * kTileWords + static_cast<size_t>(p.num_nodes) * kTileWords + p.E);
    size_t smem_rows = 4 * (static_cast<size_t>(p.R) + 1 + 2 * static_cast<size_t>(p.R) * kTileWords);
    if (p.expanded_row) smem_rows += 4 * static_cast<size_t>(p.E);       // expert bases
    if (p.node_row) smem_rows += 4 * static_cast<size_t>(p.num_nodes);   // node bases
    // node rows, then expanded rows, reuse the same region after those
    size_t extra = 0;
    if (p.node_row) extra = 4 * (2 * static_cast<size_t>(kTileWords) * p.num_nodes);
    if (p.expanded_row) {
        const size_t ex = 4 * (static_cast<size_t>(kTileTokens) * p.K +
                               2 * static_cast<size_t>(tiled_rank_warps(p.E)) * static_cast<size_t>(p.E));
        if (ex > extra) extra = ex;
    }
    smem_rows += extra;
    const int grid_tiles = p.num_tiles > 0 ? p.num_tiles : 1;
    cudaError_t e = launch_pdl(layout_count_kernel, dim3(grid_tiles), dim3(kThreads), smem_count, stream, p);
    if (e != cudaSuccess) return e;
    const int n_cols = p.R + p.E + p.num_nodes;
    const int scan_blocks = (n_cols * 32 + kThreads - 1) / kThreads;
    e = launch_pdl(layout_scan_kernel, dim3(scan_blocks), dim3(kThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(layout_rows_kernel, dim3(grid_tiles), dim3(kThreads), smem_rows, stream, p);
}

}  // namespace epg
