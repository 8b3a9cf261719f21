// Dispatch: scatter each token row once per destination rank into the
// rank-contiguous receive rows, with the token's top-k indices remapped to
// the receiving rank's local experts, its weights and its source index
// ("DeepEP Symmetric Memory" sections 6.1 and 9.2; "DeepEP V2 ElasticBuffer
// architecture", TokenLayout fragment).
//
// bf16 path (pure copy, HBM-bound, writes ~n(t) times the reads), default:
//   one CTA of 256 threads per (token, piece of <= 16 KB).  Every thread first
//   issues its 16-byte streaming loads of the piece (up to 4), then each warp
//   reads the token's destination rows itself (one lane per rank, ballot; no
//   block barrier) and stores its vectors to every destination row; warps 1,
//   2, 3 write the three per-row metadata arrays.  Thousands of short CTAs let
//   the block scheduler balance the uneven fan-out n(t).  L2: while the layout
//   kernel runs, the first wave prefetches x evict-last (all of it at
//   DeepSeek-V3 sizes) and the rows are stored evict-first.
//
// bf16 alternative (EP_DISPATCH_IMPL=0): persistent CTAs whose warp 0 drives
//   the bulk-copy engine: a ring of kStages shared-memory slots, each filled by
//   one cp.async.bulk global->shared load of a token row that completes on an
//   mbarrier, then one cp.async.bulk shared->global store per destination, so
//   a row never passes through registers; warps 1-3 write the metadata.  With
//   token_offset it splits the receive rows evenly over the CTAs.  On GB300 it
//   measured ~7% slower than the register path for every stage count, piece
//   size and L2 hint tried, so it is not the default over the whole GPU; it is
//   the SM-limited mode (num_sms > 0), one CTA per SM with a 12-slot ring,
//   where it reaches the SM's store limit (~61 GB/s on GB300) that the
//   register copies miss by ~20%.
//
// FP8 path: one CTA of up to 256 threads per (token, piece of up to 64
//   128-channel blocks), barrier-free like the bf16 register path: all 16-byte loads of
//   the piece are issued first and each warp ballots the destination rows
//   itself; then each quarter-warp owns one block per round (16 channels per
//   lane), takes amax by shuffles, scales with IEEE divides and converts with
//   cvt.rn.satfinite e4m3x2, and stores a 16-byte code vector per lane and
//   the scale to every destination row.
//
// Behind the one-cluster layout kernel (ep_layout_and_dispatch) the first
// wave of either path waits for the rows-ready signal of its token's layout
// CTA instead of the layout kernel's completion (wait_rows_ready), and the
// grid's last CTA clears the signal for the next call (clear_rows_slots).
#include <climits>

#include "ep_internal.cuh"

namespace epg {
namespace {

// Compile-time tuning of the bf16 path (defaults are the measured best).
#ifndef EP_DISPATCH_STAGES
#define EP_DISPATCH_STAGES 4          // shared-memory slots per CTA
#endif
#ifndef EP_DISPATCH_STORE_DEPTH
#define EP_DISPATCH_STORE_DEPTH 2     // bulk-store groups in flight per CTA
#endif
#ifndef EP_DISPATCH_PIECE_MAX
#define EP_DISPATCH_PIECE_MAX 16384   // bytes of a row moved by one bulk copy
#endif
#ifndef EP_DISPATCH_BALANCED
#define EP_DISPATCH_BALANCED 1        // split rows evenly when token_offset is given
#endif
#ifndef EP_DISPATCH_EVICT_FIRST
#define EP_DISPATCH_EVICT_FIRST 0     // L2 evict-first hint on the receive-row stores
#endif
#ifndef EP_ROWS_SIGNAL
#define EP_ROWS_SIGNAL 3              // rows-ready signal behind the layout kernel: bit 0 bf16, bit 1 FP8
#endif
#ifndef EP_DISPATCH_IMPL
#define EP_DISPATCH_IMPL 1            // 1: 16-byte register copies, 0: bulk-copy engine
#endif
// bf16 register path and L2: the CTAs of the first wave prefetch x into L2
// before their wait, as many generations of pieces as fit
// EP_DISPATCH_PREFETCH_L2_BYTES (all of x for DeepSeek-V3 sizes: 59 MB read
// while the layout kernel leaves HBM idle), with the evict-last policy; the
// receive rows are stored evict-first, so the 311 MB of writes stream past
// the prefetched rows instead of evicting them; a read piece of x goes back
// to the normal priority.  DS-V3 layout + dispatch 65.6 -> 61.1 us.
#ifndef EP_DISPATCH_STORE_CS
#define EP_DISPATCH_STORE_CS 2        // register path: 0 plain, 1 streaming (.cs), 2 L2 evict-first stores
#endif
#ifndef EP_DISPATCH_PREFETCH_EVICT_LAST
#define EP_DISPATCH_PREFETCH_EVICT_LAST 1
#endif
#ifndef EP_DISPATCH_PREFETCH_L2_BYTES
#define EP_DISPATCH_PREFETCH_L2_BYTES (64ll << 20)
#endif
#ifndef EP_DISPATCH_PREFETCH_MAX_GENS
#define EP_DISPATCH_PREFETCH_MAX_GENS 16
#endif
#ifndef EP_DISPATCH_FP8_L2
#define EP_DISPATCH_FP8_L2 0   // FP8 rank-row path: the same L2 policy (code stores evict-first)
#endif
#ifndef EP_DISPATCH_FP8_MIN_BLOCKS
#define EP_DISPATCH_FP8_MIN_BLOCKS 4      // FP8 path: __launch_bounds__ minimum resident CTAs per SM
#endif
#ifndef EP_DISPATCH_PREFETCH
#define EP_DISPATCH_PREFETCH 2   // FP8: x pieces a CTA of the first wave prefetches into L2 before its wait
#endif
#ifndef EP_DISPATCH_FP8_WIDE_MIN_BLOCKS
#define EP_DISPATCH_FP8_WIDE_MIN_BLOCKS 5   // same, many-token rank-row mode (fits 48 registers unspilled)
#endif
#ifndef EP_DISPATCH_FP8_HOISTED
#define EP_DISPATCH_FP8_HOISTED 1         // FP8 many-token mode: store pass with offsets hoisted out of the loop
#endif
#ifndef EP_DISPATCH_FP8_FIT_WARPS
#define EP_DISPATCH_FP8_FIT_WARPS 1       // FP8 many-token mode: CTA warps fitted to the piece's blocks
#endif
#ifndef EP_DISPATCH_FP8_PIECE_BLOCKS
#define EP_DISPATCH_FP8_PIECE_BLOCKS 64   // FP8 path: 128-channel blocks per piece (<= 64)
#endif

constexpr int kBf16Threads = 128;
constexpr int kBulkStages = EP_DISPATCH_STAGES;
constexpr int kBulkStoreDepth = EP_DISPATCH_STORE_DEPTH;
// SM-limited mode: one persistent CTA per SM whose shared-memory ring keeps
// 12 row loads in flight (a CTA's stores are bounded by the SM's write port,
// ~61 GB/s on GB300, which this ring reaches; register copies reach ~50).
constexpr int kSmBulkStages = 12;
constexpr int kSmBulkStoreDepth = 4;

// The work of one CTA.  Strided mode: items first, first + stride, ... of the
// (token, piece) list, every destination stored.  Balanced mode (rows
// numbered token by token are known, one piece per token): the CTA owns rows
// [lo, hi) of that numbering, N / gridDim rows each, and the consecutive
// tokens first .. first + count - 1 that hold them; only destinations whose
// row number falls in [lo, hi) are stored by this CTA.
// Warps (1 .. kMetaWarps) of a one-token item that write its receive
// metadata: 3 puts recv_topk_idx, recv_topk_weights and recv_src_idx on
// warps 1, 2, 3 (the chain of loads and stores a CTA's lifetime waits for
// is a third as long), 1 puts all three on warp 1.
#ifndef EP_DISPATCH_META_WARPS
#define EP_DISPATCH_META_WARPS 3
#endif
constexpr int kMetaWarps = EP_DISPATCH_META_WARPS == 1 ? 1 : 3;

struct CtaWork {
    int64_t first, count, stride;
    int lo, hi;
    int balanced;
};

// Largest t in [0, T) with a[t] <= v, for a non-decreasing a with a[0] <= v,
// searched by one warp in a 128-entry window around `guess` (one round trip of
// loads); a binary search covers a guess that misses.
__device__ int warp_last_le(const int32_t* a, int T, int v, int guess, int lane) {
    int w0 = guess - 64;
    if (w0 > T - 128) w0 = T - 128;
    if (w0 < 0) w0 = 0;
    int vals[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int idx = w0 + q * 32 + lane;
        vals[q] = idx < T ? a[idx] : INT32_MAX;
    }
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) cnt += __popc(__ballot_sync(0xffffffffu, vals[q] <= v));
    if (cnt >= 1 && (cnt < 128 || w0 + 128 >= T)) return w0 + cnt - 1;
    int res = 0;
    if (lane == 0) {
        int lo = 0, hi = T - 1;
        while (lo < hi) {
            const int mid = lo + (hi - lo + 1) / 2;
            if (a[mid] <= v) lo = mid;
            else hi = mid - 1;
        }
        res = lo;
    }
    return __shfl_sync(0xffffffffu, res, 0);
}

__device__ void cta_work(const DispatchParams& p, int lane, CtaWork& w) {
    const int64_t num_items = static_cast<int64_t>(p.T) * p.chunks;
    if (!EP_DISPATCH_BALANCED || p.token_offset == nullptr || p.chunks != 1) {
        w.balanced = 0;
        w.first = blockIdx.x;
        w.stride = gridDim.x;
        w.count = w.first < num_items ? (num_items - w.first + w.stride - 1) / w.stride : 0;
        w.lo = INT32_MIN;
        w.hi = INT32_MAX;
        return;
    }
    w.balanced = 1;
    w.stride = 1;
    const int N = EP_IN(p.T, p.T + 1) ? p.token_offset[p.T] : 0;
    const int64_t G = gridDim.x, b = blockIdx.x;
    w.lo = static_cast<int>(b * N / G);
    w.hi = static_cast<int>((b + 1) * N / G);
    if (w.lo >= w.hi) {
        w.first = 0;
        w.count = 0;
        return;
    }
    const int g0 = static_cast<int>(static_cast<int64_t>(w.lo) * p.T / N);
    const int g1 = static_cast<int>(static_cast<int64_t>(w.hi - 1) * p.T / N);
    const int t0 = warp_last_le(p.token_offset, p.T, w.lo, g0, lane);
    const int t1 = warp_last_le(p.token_offset, p.T, w.hi - 1, g1, lane);
    w.first = t0;
    w.count = t1 - t0 + 1;
}

// Metadata of token t for every destination row this CTA owns (one warp).
__device__ __forceinline__ void write_metadata(const DispatchParams& p, int t, int lane,
                                               const CtaWork& w, int part = -1) {
    const int K = p.K;
    // part -1: every array; 0: recv_topk_idx, 1: recv_topk_weights, 2: recv_src_idx only
    const bool want_idx = part < 0 || part == 0, want_w = part < 0 || part == 1, want_src = part < 0 || part == 2;
    const int64_t e_l = (lane < K && (want_idx || want_w) &&
                         EP_IN(static_cast<int64_t>(t) * K + lane, static_cast<int64_t>(p.T) * K))
                            ? p.topk_idx[static_cast<int64_t>(t) * K + lane]
                            : -1;
    const float w_l = (lane < K && want_w && p.recv_topk_weights && EP_IN(static_cast<int64_t>(t) * K + lane, static_cast<int64_t>(p.T) * K))
                          ? p.topk_weights[static_cast<int64_t>(t) * K + lane]
                          : 0.0f;
    const int tok_off = (w.balanced && EP_IN(t, p.T + 1)) ? p.token_offset[t] : 0;
    // the rank of this lane's expert and its index there, once (not per destination)
    const int e_rank = (e_l >= 0 && e_l < p.E) ? static_cast<int>(e_l) / p.experts_per_rank : -1;
    const int32_t e_local = static_cast<int32_t>(e_l) - e_rank * p.experts_per_rank;
    int m_base = 0;
    for (int rb = 0; rb < p.R; rb += 32) {
        const int r = rb + lane;
        const int d = (r < p.R && EP_IN(static_cast<int64_t>(t) * p.R + r, static_cast<int64_t>(p.T) * p.R))
                          ? p.dst_row[static_cast<int64_t>(t) * p.R + r]
                          : -1;
        (void)EP_ROW_OK(d);
        const unsigned members = __ballot_sync(0xffffffffu, d >= 0);
        const int row_tm = tok_off + m_base + __popc(members & ((1u << lane) - 1u));
        m_base += __popc(members);
        const bool mine = d >= 0 && row_tm >= w.lo && row_tm < w.hi && d < p.capacity;
        unsigned m = __ballot_sync(0xffffffffu, mine);
        while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const int64_t dd = __shfl_sync(0xffffffffu, d, src);
            const int rr = rb + src;
            if (lane < K && EP_IN(dd * K + lane, p.capacity * K)) {
                const bool on = e_rank == rr;
                if (want_idx && p.recv_topk_idx)
                    p.recv_topk_idx[dd * K + lane] =
                        on ? e_local : -1;
                if (want_w && p.recv_topk_weights) p.recv_topk_weights[dd * K + lane] = on ? w_l : 0.0f;
            }
            if (want_src && lane == 0 && p.recv_src_idx && EP_IN(dd, p.capacity)) p.recv_src_idx[dd] = t;
        }
    }
}

template <int kStages, int kStoreDepth>
__global__ void __launch_bounds__(kBf16Threads) dispatch_bf16_kernel(const DispatchParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ CtaWork s_work;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    uint8_t* stage = smem + 128;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t row_bytes = static_cast<uint32_t>(p.H) * 2u;
    pdl_wait();

    if (warp == 0) {
        CtaWork w;
        cta_work(p, lane, w);
        if (lane == 0) {
            s_work = w;
            for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
            fence_mbar_init();
        }
    }
    __syncthreads();
    const CtaWork w = s_work;
    const int64_t my_n = w.count;

    if (warp == 0) {
#if EP_DISPATCH_EVICT_FIRST
        const uint64_t policy = l2_policy_evict_first();
#endif
        int64_t issued = 0;  // lane 0 only
        auto issue = [&](int64_t i) {
            const int64_t it = w.first + i * w.stride;
            const int64_t t = it / p.chunks;
            const uint32_t off = static_cast<uint32_t>(it - t * p.chunks) * p.chunk_bytes;
            const uint32_t bytes = min(p.chunk_bytes, row_bytes - off);
            const int slot = static_cast<int>(i % kStages);
            mbar_arrive_expect_tx(&bars[slot], bytes);
#if EP_GET_CHECKED
            // an out-of-range piece is not loaded; its wait then runs out
            // (bounded) and the CTA winds down
            if (!EP_IN_BYTES(t * row_bytes + off, bytes, static_cast<int64_t>(p.T) * row_bytes)) return;
#endif
#ifdef EP_TEST_DROP_FIRST_LOAD
            // failure-path test build only: CTA 0 announces its first load
            // and never issues it, so that slot's wait runs out (no copy is
            // in flight for it, every access stays in bounds)
            if (blockIdx.x == 0 && i == 0) return;
#endif
            bulk_load(stage + static_cast<size_t>(slot) * p.chunk_bytes, p.x + t * row_bytes + off,
                      bytes, &bars[slot]);
        };
        if (lane == 0) {
            for (; issued < kStages && issued < my_n; ++issued) issue(issued);
        }
        bool ok = true;
        bool cap_bad = false;
        int64_t i = 0;
        for (; i < my_n; ++i) {
            const int slot = static_cast<int>(i % kStages);
            const int64_t it = w.first + i * w.stride;
            const int64_t t = it / p.chunks;
            const uint32_t off = static_cast<uint32_t>(it - t * p.chunks) * p.chunk_bytes;
            const uint32_t bytes = min(p.chunk_bytes, row_bytes - off);
            // destination rows of the first 32 ranks and the token's first row
            // number: loaded before the wait so their latency overlaps it
            const int64_t n_tr = static_cast<int64_t>(p.T) * p.R;
            const int d0 = (lane < p.R && EP_IN(t * p.R + lane, n_tr)) ? p.dst_row[t * p.R + lane] : -1;
            const int tok_off = (w.balanced && EP_IN(t, p.T + 1)) ? p.token_offset[t] : 0;
            const bool landed = mbar_wait_bounded(&bars[slot], static_cast<uint32_t>((i / kStages) & 1));
            if (!__all_sync(0xffffffffu, landed)) {
                ok = false;
                break;
            }
            const uint8_t* src = stage + static_cast<size_t>(slot) * p.chunk_bytes;
            int m_base = 0;
            for (int rb = 0; rb < p.R; rb += 32) {
                const int r = rb + lane;
                const int d = rb == 0 ? d0 : ((r < p.R && EP_IN(t * p.R + r, n_tr)) ? p.dst_row[t * p.R + r] : -1);
                (void)EP_ROW_OK(d);
                const unsigned members = __ballot_sync(0xffffffffu, d >= 0);
                const int row_tm = tok_off + m_base + __popc(members & ((1u << lane) - 1u));
                m_base += __popc(members);
                if (d >= 0 && row_tm >= w.lo && row_tm < w.hi) {
                    if (d < p.capacity &&
                        EP_IN_BYTES(static_cast<int64_t>(d) * row_bytes + off, bytes, p.capacity * row_bytes)) {
#if EP_DISPATCH_EVICT_FIRST
                        bulk_store_evict_first(p.recv_x + static_cast<int64_t>(d) * row_bytes + off, src,
                                               bytes, policy);
#else
                        bulk_store(p.recv_x + static_cast<int64_t>(d) * row_bytes + off, src, bytes);
#endif
                    }
                    else
                        cap_bad = true;
                }
            }
            bulk_commit();
            bulk_wait_read<kStoreDepth - 1>();
            __syncwarp();
            const int64_t j = i - (kStoreDepth - 1);
            if (lane == 0 && j >= 0 && j + kStages < my_n) {
                issue(j + kStages);
                ++issued;
            }
        }
        bulk_wait_all<0>();
        if (!ok) {
            // Drain the loads still in flight (bounded) before shared memory is released.
            if (lane == 0) {
                for (int64_t k = i; k < issued; ++k)
                    mbar_wait_bounded(&bars[k % kStages], static_cast<uint32_t>((k / kStages) & 1));
                atomicOr(p.status, EP_ERR_TIMEOUT);
            }
        }
        if (__any_sync(0xffffffffu, cap_bad) && lane == 0) atomicOr(p.status, EP_ERR_CAPACITY);
    } else {
        // Metadata: this CTA's tokens (piece 0 of each), round-robin over warps 1..3.
        const int mw = warp - 1;
        const int n_mw = kBf16Threads / 32 - 1;
        int64_t count = 0;
        for (int64_t i = 0; i < my_n; ++i) {
            const int64_t it = w.first + i * w.stride;
            if (it % p.chunks != 0) continue;
            if ((count++ % n_mw) != mw) continue;
            write_metadata(p, static_cast<int>(it / p.chunks), lane, w);
        }
    }
}

// Expanded mode metadata of token t (one warp, lane k): every valid (t, k)
// row gets the source token and the weight of that top-k slot.
__device__ __forceinline__ void write_expanded_metadata(const DispatchParams& p, int t, int lane) {
    if (lane >= p.K) return;
    const int64_t ek = static_cast<int64_t>(t) * p.K + lane, n_tk = static_cast<int64_t>(p.T) * p.K;
    if (!EP_IN(ek, n_tk)) return;
    const int d = p.expanded_row[ek];
    (void)EP_ROW_OK(d);
    if (d < 0 || d >= p.capacity) return;
    if (p.recv_src_idx) p.recv_src_idx[d] = t;
    if (p.recv_weight) p.recv_weight[d] = p.topk_weights[ek];
}

// Before waiting on the previous kernel (normally the layout, which leaves
// HBM idle for several microseconds), thread 0 of a first-wave CTA asks L2 to
// fetch the x pieces of its own item and of the items that will follow on
// the same slot (b + j * prefetch_ctas).  A prefetch only fills L2, the
// coherence point, and x is still read after the wait, so a producer of x
// that is still running cannot make the kernel read stale data.
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes, bool evict_last = false) {
    if (evict_last)
        asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(ptr), "r"(bytes),
                     "l"(l2_policy_evict_last())
                     : "memory");
    else
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// FP8 (latency-bound): later CTAs keep the distance, CTA b >= prefetch_ctas
// fetching the piece of item b + (prefetch_items - 1) * prefetch_ctas, one
// generation ahead (DS-V3 39.9 -> 38.1 us).  The bf16 copy, bound by HBM
// writes, lost 2-6% to that extra L2 traffic, so there only the first wave
// prefetches: every generation that fits the L2 budget, evict-last (see
// EP_DISPATCH_PREFETCH_EVICT_LAST).
template <bool kFp8>
__device__ __forceinline__ void prefetch_x(const DispatchParams& p) {
    if (threadIdx.x != 0 || p.prefetch_items <= 0) return;
    const uint32_t row_bytes = static_cast<uint32_t>(p.H) * 2u;
    const uint32_t piece = kFp8 ? static_cast<uint32_t>(p.chunk_blocks) * 256u : p.chunk_bytes;
    const int64_t n_items = static_cast<int64_t>(p.T) * p.chunks;
    const int64_t b = blockIdx.x, g = p.prefetch_ctas;
    const int j0 = b < g ? 0 : ((kFp8 && !p.prefetch_evict_last) ? p.prefetch_items - 1 : p.prefetch_items);
    for (int j = j0; j < p.prefetch_items; ++j) {
        const int64_t it = b + static_cast<int64_t>(j) * g;
        if (it >= n_items) return;
        const int t = static_cast<int>(it / p.chunks);
        const uint32_t off = static_cast<uint32_t>(it - static_cast<int64_t>(t) * p.chunks) * piece;
        prefetch_l2(p.x + static_cast<int64_t>(t) * row_bytes + off, min(piece, row_bytes - off),
                    p.prefetch_evict_last != 0);
    }
}

// Few-token layout inside the dispatch (ep_layout_and_dispatch): each CTA
// derives the destination row of its token on every rank from topk_idx
// alone, as the layout defines it ("DeepEP Symmetric Memory" section 6.1:
// the per-rank prefix sum of received tokens plus the destination slot
// index):
//   dst_row[t, r] = rank_offset[r] + #{t' < t : t' has an expert on r},
//   rank_offset = exclusive prefix of the per-rank token counts,
// with masked (-1) and invalid ids counting for no rank, so no layout kernel
// has to run first.  The CTA of piece 0 of token t also writes the token's
// layout rows (dst_row, is_token_in_rank, token_offset[t]).  Two extra CTAs
// of the grid (kLayoutCta, no dispatch work; c selects the part) write the
// counts and offsets beside the dispatch CTAs: part 0 per rank, per node,
// src_dst_count, rank_offset and token_offset[T]; part 1 per expert with
// the alignment and expert_offset, and flags invalid ids.  CTA-wide: every
// thread calls it, with blockDim.x == 256, T <= kSelfMaxTokens, R <= 32,
// K <= kSelfMaxTopk and E <= kSelfMaxExperts.  Returns in lane r of every
// warp the row of rank r for token t, or -1 (dispatch CTAs).
constexpr int kSelfMaxTokens = kSelfRouteMaxTokens;
constexpr int kSelfMaxTopk = kSelfRouteMaxTopk;
constexpr int kSelfMaxExperts = kSelfRouteMaxExperts;
// Layout CTAs after the dispatch items: the last writes the per-rank counts
// and offsets, src_dst_count and the per-node counts; the one before it the
// per-expert counts and offsets (and flags invalid ids).
constexpr int kSelfLayoutCtas = 2;
static_assert(kSelfMaxTokens <= 256, "self_route_layout: one thread per token in a 256-thread CTA");
struct SelfRouteSmem {
    uint32_t mask[kSelfMaxTokens];           // ranks holding each token (bit r)
    uint32_t bal[kSelfMaxTokens / 32][32];   // [word of 32 tokens][rank]: membership bits
    int hist[kSelfMaxExperts];               // expert layout CTA: entries per expert, then offsets in the chunk
    int chunk[kSelfMaxExperts / 32];         // expert layout CTA: aligned entries per 32 experts, then their prefix
};

// The CTA's one SelfRouteSmem (a function-scope __shared__ object exists
// once per CTA), shared by the dispatch items and the layout CTA.
__device__ __forceinline__ SelfRouteSmem& self_smem() {
    __shared__ SelfRouteSmem s;
    return s;
}

#ifndef EP_SELF_ROUTE_COALESCED
#define EP_SELF_ROUTE_COALESCED 1   // 16-byte top-k loads in the dispatch CTAs' routing step
#endif
#ifndef EP_SELF_META_PIECE
#define EP_SELF_META_PIECE 1        // piece whose last warps write the receive metadata (fewer than four pieces)
#endif
#ifndef EP_SELF_META_SPREAD
#define EP_SELF_META_SPREAD 1       // with four or more pieces, one metadata array per piece
#endif
#ifndef EP_SELF_EARLY_META
#define EP_SELF_EARLY_META 1        // that warp loads the token's entries before the routing step
#endif

template <bool kLayoutCta>
__device__ int self_route_layout(const DispatchParams& p, int t, int c, SelfRouteSmem& s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr bool cta0 = kLayoutCta;
    // layout CTAs: c is the part (0: ranks, 1: experts); CTA-uniform
    const bool rank_part = !cta0 || c == 0;
    const bool expert_part = cta0 && c == 1;
    int64_t e[kSelfMaxTopk];
    // K in {2, 4, 8, 16} and a 16-byte aligned topk_idx: 16-byte loads (two
    // entries each) over the whole [T, K] block, and the K / 2 lanes of a
    // token OR their rank bits together (a quarter of the L2 requests of one
    // thread per token, on a block that every CTA reads).  Thread tid holds
    // entries 2 (j * 256 + tid) and the next in e[2 j], e[2 j + 1].
    const int q = p.K >> 1;
    const bool coalesced = EP_SELF_ROUTE_COALESCED && (p.K & (p.K - 1)) == 0 && p.K >= 2 &&
                           (reinterpret_cast<uintptr_t>(p.topk_idx) & 15u) == 0;
    const int n_pairs = p.T * q;
    if (coalesced) {
        static_assert(kSelfMaxTokens * kSelfMaxTopk / 2 <= 256 * (kSelfMaxTopk / 2), "entry pairs per thread");
#pragma unroll
        for (int j = 0; j < kSelfMaxTopk / 2; ++j) {
            const int i = j * 256 + tid;   // blockDim.x == 256
            e[2 * j] = e[2 * j + 1] = -1;
            if (j * 256 >= n_pairs) continue;   // the same trips in every lane
            uint32_t m = 0;
            if (i < n_pairs && EP_IN(2 * static_cast<int64_t>(i) + 1, static_cast<int64_t>(p.T) * p.K)) {
                const longlong2 v = *reinterpret_cast<const longlong2*>(p.topk_idx + 2 * static_cast<int64_t>(i));
                e[2 * j] = v.x;
                e[2 * j + 1] = v.y;
                if (v.x >= 0 && v.x < p.E) m |= 1u << (static_cast<int>(v.x) / p.experts_per_rank);
                if (v.y >= 0 && v.y < p.E) m |= 1u << (static_cast<int>(v.y) / p.experts_per_rank);
            }
            for (int o = 1; o < q; o <<= 1) m |= __shfl_xor_sync(0xffffffffu, m, o);
            if (i < n_pairs && (i & (q - 1)) == 0) s.mask[i / q] = m;
        }
    } else if (tid < p.T) {   // one thread per token: all K entries in flight at once
#pragma unroll
        for (int k = 0; k < kSelfMaxTopk; ++k) {
            const int64_t i = static_cast<int64_t>(tid) * p.K + k;
            e[k] = (k < p.K && EP_IN(i, static_cast<int64_t>(p.T) * p.K)) ? p.topk_idx[i] : -1;
        }
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < kSelfMaxTopk; ++k)
            if (e[k] >= 0 && e[k] < p.E) m |= 1u << (static_cast<int>(e[k]) / p.experts_per_rank);
        s.mask[tid] = m;
    }
    if (expert_part)
        for (int i = tid; i < p.E; i += blockDim.x) s.hist[i] = 0;
    __syncthreads();
    if (expert_part && (coalesced || tid < p.T)) {   // every entry once: the expert histogram, invalid ids
        bool bad = false;
#pragma unroll
        for (int k = 0; k < kSelfMaxTopk; ++k) {
            if (!coalesced && k >= p.K) break;
            if (e[k] >= 0 && e[k] < p.E) atomicAdd(&s.hist[e[k]], 1);
            else if (e[k] != -1) bad = true;
        }
        if (bad) atomicOr(p.status, EP_ERR_INVALID_INDEX);
    }
    const int n_words = (p.T + 31) >> 5;
    if (rank_part && warp < n_words) {
        const int j = (warp << 5) + lane;
        const uint32_t m = j < p.T ? s.mask[j] : 0u;
        for (int r = 0; r < p.R; ++r) {
            const uint32_t b = __ballot_sync(0xffffffffu, (m >> r) & 1u);
            if (lane == r) s.bal[warp][r] = b;
        }
    }
    __syncthreads();
    int total = 0, before = 0;
    if (rank_part && lane < p.R) {
        const int tw = t >> 5;
        for (int w = 0; w < n_words; ++w) {
            const uint32_t b = s.bal[w][lane];
            total += __popc(b);
            if (w < tw) before += __popc(b);
            else if (w == tw) before += __popc(b & ((1u << (t & 31)) - 1u));
        }
    }
    const int incl = warp_inclusive_scan(total);   // lanes >= R add 0
    const int offset = incl - total;
    const bool in = lane < p.R && ((s.mask[t] >> lane) & 1u);
    const int d = in ? offset + before : -1;

    // the token's layout rows, one array per warp: on this short grid the
    // first store into each array waits for its address translation, and on
    // separate warps those waits overlap
    if (!kLayoutCta && c == 0 && warp < 3) {
        const int64_t tr = static_cast<int64_t>(t) * p.R + lane;
        const bool ok = lane < p.R && EP_IN(tr, static_cast<int64_t>(p.T) * p.R);
        if (warp == 0) {
            if (ok) p.l_dst_row[tr] = d;
        } else if (warp == 1) {
            if (ok) p.l_is_token_in_rank[tr] = in ? 1 : 0;
        } else {
            const int rows_before = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(before)));
            if (lane == 0 && p.l_token_offset && EP_IN(t, p.T + 1)) p.l_token_offset[t] = rows_before;
        }
    }
    if (cta0 && rank_part) {
        const int n_rows = __shfl_sync(0xffffffffu, incl, 31);
        if (warp == 0) {
            if (lane < p.R && EP_IN(lane, p.R)) {
                p.l_num_tokens_per_rank[lane] = total;
                p.l_rank_offset[lane] = offset;
            }
            if (lane == 0) {
                if (EP_IN(p.R, p.R + 1)) p.l_rank_offset[p.R] = n_rows;
                if (p.l_token_offset && EP_IN(p.T, p.T + 1)) p.l_token_offset[p.T] = n_rows;
            }
        }
        // src_dst_count[src][r]: tokens of source rank src (T / R each) on rank r
        if (p.l_src_dst_count) {
            const int per_src = p.T / p.R;
            for (int j = tid; j < p.R * p.R; j += blockDim.x) {
                const int src = j / p.R, r = j - src * p.R;
                int cnt = 0;
                for (int u = src * per_src; u < (src + 1) * per_src; ++u) cnt += (s.mask[u] >> r) & 1u;
                if (EP_IN(j, p.R * p.R)) p.l_src_dst_count[j] = cnt;
            }
        }
        // tokens reaching each node (ranks [n * rpn, (n + 1) * rpn))
        if (p.l_num_tokens_per_node) {
            for (int n = tid; n < p.l_num_nodes; n += blockDim.x) {
                // a token reaches node n when any rank of n holds it: OR the
                // ranks' membership words, count the bits
                int cnt = 0;
                for (int w = 0; w < n_words; ++w) {
                    uint32_t o = 0u;
                    for (int r = n * p.l_ranks_per_node; r < (n + 1) * p.l_ranks_per_node; ++r) o |= s.bal[w][r];
                    cnt += __popc(o);
                }
                if (EP_IN(n, p.l_num_nodes)) p.l_num_tokens_per_node[n] = cnt;
            }
        }
    }
    if (expert_part) {
        // per-expert counts, rounded up to the alignment, scanned
        const int n_chunks = (p.E + 31) >> 5;
        for (int ch = warp; ch < n_chunks; ch += blockDim.x >> 5) {
            const int ex = ch * 32 + lane;
            const int cnt = ex < p.E ? s.hist[ex] : 0;
            if (ex < p.E && EP_IN(ex, p.E)) p.l_num_tokens_per_expert[ex] = cnt;
            const int al = (cnt + p.l_alignment - 1) / p.l_alignment * p.l_alignment;
            const int ci = warp_inclusive_scan(al);
            if (ex < p.E) s.hist[ex] = ci - al;
            if (lane == 31) s.chunk[ch] = ci;
        }
        __syncthreads();   // CTA-uniform branch
        if (warp == 0) {   // exclusive prefix of the chunk totals (at most 64 chunks)
            const int a = lane < n_chunks ? s.chunk[lane] : 0;
            const int b = 32 + lane < n_chunks ? s.chunk[32 + lane] : 0;
            const int ia = warp_inclusive_scan(a);
            const int ib = warp_inclusive_scan(b) + __shfl_sync(0xffffffffu, ia, 31);
            if (lane < n_chunks) s.chunk[lane] = ia - a;
            if (32 + lane < n_chunks) s.chunk[32 + lane] = ib - b;
            if (lane == 31 && EP_IN(p.E, p.E + 1)) p.l_expert_offset[p.E] = ib;
        }
        __syncthreads();
        for (int ex = tid; ex < p.E; ex += blockDim.x)
            if (EP_IN(ex, p.E + 1)) p.l_expert_offset[ex] = s.chunk[ex >> 5] + s.hist[ex];
    }
    return d;
}

// The token's top-k entries for its receive metadata, loaded where the
// call stands (volatile: issued before the routing step, not sunk to the use).
__device__ __forceinline__ void load_token_entries(const DispatchParams& p, int t, int lane, int64_t& e_l, float& w_l) {
    const int64_t ek = static_cast<int64_t>(t) * p.K + lane, n_tk = static_cast<int64_t>(p.T) * p.K;
    e_l = -1;
    w_l = 0.0f;
    if (lane < p.K && EP_IN(ek, n_tk)) {
        asm volatile("ld.global.nc.s64 %0, [%1];" : "=l"(e_l) : "l"(p.topk_idx + ek));
        if (p.recv_topk_weights) asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(w_l) : "l"(p.topk_weights + ek));
    }
}

// The self-routed item's piece whose warps write the token's receive
// metadata: piece 1 when there is one, so that piece 0 (which writes the
// token's layout rows) and it each carry one extra chain of first touches.
__device__ __forceinline__ int self_meta_piece(const DispatchParams& p) {
    return EP_SELF_META_PIECE < p.chunks ? EP_SELF_META_PIECE : p.chunks - 1;
}

// Which receive-metadata part (0..2) warp warp_g (of nw) of piece c
// writes, or -1.  The last warps take it: on the few-token FP8 grid the last
// warp has no blocks of the piece to cast, so the metadata overlaps the
// other warps' stores.  With at least four pieces each part has a piece of
// its own (pieces 1, 2, 3, last warp); otherwise the last three warps of the
// metadata piece write one part each.
__device__ __forceinline__ int self_meta_part(const DispatchParams& p, int c, int warp_g, int nw) {
    if (EP_SELF_META_SPREAD && p.chunks >= 4) return (warp_g == nw - 1 && c >= 1 && c <= 3) ? c - 1 : -1;
    const int part = warp_g - (nw - 3);
    return (c == self_meta_piece(p) && part >= 0 && part < 3) ? part : -1;
}

// One of the token's receive-metadata arrays (part 0: recv_topk_idx, 1:
// recv_topk_weights, 2: recv_src_idx) for every destination (lane r of d:
// rank r's row, R <= 32); one warp per part, so that the first stores into
// the three arrays wait for their address translations side by side.  Same
// entries as write_metadata.
__device__ __forceinline__ void write_metadata_part(const DispatchParams& p, int t, int lane, int d, int64_t e_l,
                                                    float w_l, int part) {
    const int K = p.K;
    // the rank of this lane's expert and its index there, once (not per destination)
    const int e_rank = (e_l >= 0 && e_l < p.E) ? static_cast<int>(e_l) / p.experts_per_rank : -1;
    const int32_t e_local = static_cast<int32_t>(e_l) - e_rank * p.experts_per_rank;
    unsigned m = __ballot_sync(0xffffffffu, d >= 0 && d < p.capacity);
    while (m) {
        const int rr = __ffs(m) - 1;
        m &= m - 1;
        const int64_t dd = __shfl_sync(0xffffffffu, d, rr);
        if (part < 2) {
            if (lane < K && EP_IN(dd * K + lane, p.capacity * K)) {
                const bool on = e_rank == rr;
                if (part == 0) {
                    if (p.recv_topk_idx)
                        p.recv_topk_idx[dd * K + lane] = on ? e_local : -1;
                } else if (p.recv_topk_weights) {
                    p.recv_topk_weights[dd * K + lane] = on ? w_l : 0.0f;
                }
            }
        } else if (lane == 0 && p.recv_src_idx && EP_IN(dd, p.capacity)) {
            p.recv_src_idx[dd] = t;
        }
    }
}

// Rows-ready wait (ep_layout_and_dispatch, cluster layout): thread 0 polls
// the slot of the layout CTA that writes token t's rows until it holds the
// call's tag, or waits for the layout kernel's completion after kRowsWaitNs,
// then counts itself as a reader of the slot (a relaxed add that returns
// nothing, so no wait: the count only tells the last CTA when it may clear
// the tag, and a tag cleared early costs a reader the fallback, never a
// wrong row); the CTA's barrier then releases the row loads, which are plain
// loads: the layout CTA's release, this acquire and the barrier order them
// after the rows' stores.  Every first-wave CTA calls this exactly once.
__device__ __forceinline__ void wait_rows_ready(const DispatchParams& p, int t) {
    if (threadIdx.x == 0) {
        const int c = t / p.rows_tokens;
        bool seen = false;
        uint64_t* slot = p.rows_ready + static_cast<size_t>(c) * kReadyWords;
        const bool ok = EP_IN(c, p.rows_slots);
        if (ok) {
            const uint64_t start = global_timer_ns();
            while (!(seen = ld_acquire_u64(slot) == p.rows_tag)) {
                if (global_timer_ns() - start > kRowsWaitNs) break;
                __nanosleep(64);
            }
        }
        if (!seen) pdl_wait();
        if (ok) red_relaxed_add_u32(reinterpret_cast<uint32_t*>(slot + 1), 1u);
    }
    __syncthreads();
}

// The grid's last CTA, after its item: once the layout kernel has completed
// (every tag published) and each slot has counted all its readers (the CTAs
// of its tokens below rows_first_wave), clear the tags.  Should a count stay short for kRowsWaitNs
// the tag is cleared all the same: a reader that then finds none waits for
// the layout kernel's completion, which has already happened.
__device__ __forceinline__ void clear_rows_slots(const DispatchParams& p) {
    pdl_wait();
    for (int c = threadIdx.x; c < p.rows_slots; c += blockDim.x) {
        uint64_t* slot = p.rows_ready + static_cast<size_t>(c) * kReadyWords;
        const int64_t first = static_cast<int64_t>(c) * p.rows_tokens * p.chunks;
        const int64_t end = min(min(static_cast<int64_t>(c + 1) * p.rows_tokens, static_cast<int64_t>(p.T)) * p.chunks,
                                static_cast<int64_t>(p.rows_first_wave));
        const uint32_t readers = end > first ? static_cast<uint32_t>(end - first) : 0u;
        const uint64_t start = global_timer_ns();
        while (ld_acquire_u32(reinterpret_cast<const uint32_t*>(slot + 1)) < readers) {
            if (global_timer_ns() - start > kRowsWaitNs) break;
            __nanosleep(64);
        }
        *reinterpret_cast<volatile uint64_t*>(slot) = 0ull;
    }
}

constexpr int kRegThreads = 256;
constexpr int kRegUnroll = 4;
constexpr int kSelfRegBlocks = 4;   // self-routing bf16 CTAs per SM (registers for the top-k entries, no spills)

// SM-limited mode: CTAs of kSmGroups groups, one per SM, each group looping
// over (token, piece) items.
constexpr int kSmGroups = 4;

// Register path: one group of 256 threads per (token, piece); each thread
// loads up to kRegUnroll 16-byte vectors of the piece, its warp reads the
// token's destination rows (one lane per rank) and broadcasts them by
// shuffles, and the thread stores its vectors to every destination.  Warps
// never wait for one another.  kExpanded: the destinations are the token's
// expanded rows (one per valid top-k slot) instead of one row per rank.
// kGroups > 1 (SM-limited mode): several groups per CTA looping over items.
// One (token, piece) item of the register path, by one group of 256 threads.
template <bool kExpanded, bool kSelf, int kMW = kMetaWarps>
__device__ __forceinline__ void dispatch_regs_item(const DispatchParams& p, int64_t it, int gtid, int warp_g,
                                                   int lane, bool& cap_bad, bool signal = false) {
    const uint32_t row_bytes = static_cast<uint32_t>(p.H) * 2u;
    const int t = static_cast<int>(it / p.chunks);
    const int c = static_cast<int>(it - static_cast<int64_t>(t) * p.chunks);
    const uint32_t off = static_cast<uint32_t>(c) * p.chunk_bytes;
    const uint32_t bytes = min(p.chunk_bytes, row_bytes - off);
    const int nvec = static_cast<int>(bytes / 16);
    const int64_t src_off = static_cast<int64_t>(t) * row_bytes + off;   // in x (T rows)
    const int64_t x_bytes = static_cast<int64_t>(p.T) * row_bytes, rx_bytes = p.capacity * row_bytes;
    const uint8_t* src = p.x + src_off;
#if EP_DISPATCH_STORE_CS == 2
    const uint64_t store_pol = l2_policy_evict_first();
#endif
    // this thread's loads and the warp's destination rows, all in flight together
    uint4 u[kRegUnroll];
#pragma unroll
    for (int k = 0; k < kRegUnroll; ++k) {
        const int v = gtid + k * kRegThreads;
        if (v < nvec && EP_IN_BYTES(src_off + static_cast<int64_t>(v) * 16, 16, x_bytes))
            u[k] = ld_stream_v4(src + static_cast<size_t>(v) * 16);
    }
    const int n_dst = kExpanded ? p.K : p.R;
    const int64_t drow0 = static_cast<int64_t>(t) * n_dst, n_drow = static_cast<int64_t>(p.T) * n_dst;
    const int32_t* drow = (kExpanded ? p.expanded_row : p.dst_row) + drow0;
    int d0, d1;
    int64_t me_l = -1;   // self-routed: the token's entries, for the receive metadata
    float mw_l = 0.0f;
    if constexpr (kSelf) {
        if (EP_SELF_EARLY_META && static_cast<unsigned>(self_meta_part(p, c, warp_g, kRegThreads / 32)) < 2u)
            load_token_entries(p, t, lane, me_l, mw_l);
        d0 = self_route_layout<false>(p, t, c, self_smem());   // R <= 32
        d1 = -1;
    } else {
        if (signal) wait_rows_ready(p, t);   // x is already in flight
        d0 = (lane < n_dst && EP_IN(drow0 + lane, n_drow)) ? drow[lane] : -1;
        d1 = (32 + lane < n_dst && EP_IN(drow0 + 32 + lane, n_drow)) ? drow[32 + lane] : -1;   // ranks 32..63
        (void)EP_ROW_OK(d0);
        (void)EP_ROW_OK(d1);
    }
    if (kSelf) {
        const int part = self_meta_part(p, c, warp_g, kRegThreads / 32);
        if (part >= 0) {
            if (!EP_SELF_EARLY_META && part < 2) load_token_entries(p, t, lane, me_l, mw_l);
            write_metadata_part(p, t, lane, d0, me_l, mw_l, part);
        }
    } else if (c == 0 && (kExpanded ? warp_g == 1 : (warp_g >= 1 && warp_g <= kMW))) {
        if (kExpanded) {
            write_expanded_metadata(p, t, lane);
        } else {
            CtaWork all;
            all.first = 0;
            all.count = 0;
            all.stride = 1;
            all.lo = INT32_MIN;
            all.hi = INT32_MAX;
            all.balanced = 0;
            // one array per warp (kMW == 3), or all on warp 1
            write_metadata(p, t, lane, all, kMW == 3 ? warp_g - 1 : -1);
        }
    }
    for (int base = 0; base < nvec; base += kRegUnroll * kRegThreads) {
        if (base > 0) {
#pragma unroll
            for (int k = 0; k < kRegUnroll; ++k) {
                const int v = base + gtid + k * kRegThreads;
                if (v < nvec && EP_IN_BYTES(src_off + static_cast<int64_t>(v) * 16, 16, x_bytes))
                    u[k] = ld_stream_v4(src + static_cast<size_t>(v) * 16);
            }
        }
        for (int rb = 0; rb < n_dst; rb += 32) {
            const int d = rb == 0    ? d0
                          : rb == 32 ? d1
                                     : ((rb + lane < n_dst && EP_IN(drow0 + rb + lane, n_drow)) ? drow[rb + lane] : -1);
            if (rb >= 64) (void)EP_ROW_OK(d);
            if (d >= p.capacity && c == 0) cap_bad = true;
            unsigned m = __ballot_sync(0xffffffffu, d >= 0 && d < p.capacity);
            while (m) {
                const int sl = __ffs(m) - 1;
                m &= m - 1;
                const int64_t dst_off = static_cast<int64_t>(__shfl_sync(0xffffffffu, d, sl)) * row_bytes + off;
                uint8_t* dst = p.recv_x + dst_off;
#pragma unroll
                for (int k = 0; k < kRegUnroll; ++k) {
                    const int v = base + gtid + k * kRegThreads;
                    if (v < nvec && EP_IN_BYTES(dst_off + static_cast<int64_t>(v) * 16, 16, rx_bytes)) {
#if EP_DISPATCH_STORE_CS == 1
                        st_cs_v4(dst + static_cast<size_t>(v) * 16, u[k]);
#elif EP_DISPATCH_STORE_CS == 2
                        st_v4_hint(dst + static_cast<size_t>(v) * 16, u[k], store_pol);
#else
                        st_v4(dst + static_cast<size_t>(v) * 16, u[k]);
#endif
                    }
                }
            }
        }
#if EP_DISPATCH_PREFETCH_EVICT_LAST
        // These x vectors are read: the 128-byte lines they start (whole
        // lines inside x only) go back to the normal eviction priority, so
        // that x does not outlive the kernel in L2 ahead of other data.
#pragma unroll
        for (int k = 0; k < kRegUnroll; ++k) {
            const int v = base + gtid + k * kRegThreads;
            const uint8_t* a = src + static_cast<size_t>(v) * 16;
            if (v < nvec && (reinterpret_cast<uintptr_t>(a) & 127u) == 0 &&
                src_off + static_cast<int64_t>(v) * 16 + 128 <= x_bytes)
                l2_priority_normal(a);
        }
#endif
    }
}

// kSelf (ep_layout_and_dispatch, few tokens, one CTA per item): there is no
// layout kernel in front; each CTA derives its token's destination rows
// itself and writes the token's layout rows, and kSelfLayoutCtas extra CTAs
// the layout's counts and offsets (self_route_layout).
template <bool kExpanded, int kGroups, bool kSelf = false>
__global__ void __launch_bounds__(kRegThreads * kGroups, kGroups > 1 ? 1 : kSelf ? kSelfRegBlocks : 6)
    dispatch_bf16_regs_kernel(const DispatchParams p) {
    const int gtid = static_cast<int>(threadIdx.x) % kRegThreads;
    const int warp_g = gtid >> 5;   // warp within the group
    const int lane = threadIdx.x & 31;
    bool cap_bad = false;
    if (kSelf && blockIdx.x >= gridDim.x - kSelfLayoutCtas) {   // the layout's counts and offsets
        pdl_wait();
        self_route_layout<true>(p, 0, static_cast<int>(gridDim.x - 1 - blockIdx.x), self_smem());
        return;
    }
    if (kGroups == 1) prefetch_x<false>(p);
    // With the rows-ready signal (first wave) x was complete before the
    // layout kernel passed its own wait, and only dst_row waits (for the
    // signal).  Later CTAs start once the layout kernel has ended: for them
    // the wait on it costs nothing, and a poll would cost a round trip.
    const bool signal_call = kGroups == 1 && !kSelf && !kExpanded && p.rows_ready != nullptr;
    const bool signal = signal_call && static_cast<int>(blockIdx.x) < p.rows_first_wave;
    if (!signal) pdl_wait();   // before any load: the previous kernel may write x
    if (kGroups == 1) {
        dispatch_regs_item<kExpanded, kSelf>(p, blockIdx.x, gtid, warp_g, lane, cap_bad, signal);
        if (signal_call && blockIdx.x == gridDim.x - 1) clear_rows_slots(p);
    } else {
        const int64_t n_items = static_cast<int64_t>(p.T) * p.chunks;
        const int group = static_cast<int>(threadIdx.x) / kRegThreads;
        for (int64_t it = static_cast<int64_t>(blockIdx.x) * kGroups + group; it < n_items;
             it += static_cast<int64_t>(gridDim.x) * kGroups)
            dispatch_regs_item<kExpanded, false, 1>(p, it, gtid, warp_g, lane, cap_bad);
    }
    if (warp_g == 0 && __any_sync(0xffffffffu, cap_bad) && lane == 0) atomicOr(p.status, EP_ERR_CAPACITY);
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    uint16_t lo, hi;
    // cvt ... d, x, y puts x in the upper byte and y in the lower byte.
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// (a * m, b * m), each product rounded to nearest even as by a scalar
// multiply, in one packed fp32x2 instruction.
__device__ __forceinline__ float2 mul2_rn(float a, float b, uint64_t mm) {
    uint64_t x, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(mm));
    float2 y;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(y.x), "=f"(y.y) : "l"(r));
    return y;
}

constexpr int kFp8Threads = 256;
constexpr int kFp8Rounds = 2;   // rounds of blocks per item (loads of every round issued first)

// One (token, piece) FP8 item, by one group of 256 threads, barrier-free.
// kLanes lanes share one 128-channel block (each lane 128 / kLanes channels):
// 8 (two 16-byte loads and a 16-byte code store per lane, fewer instructions
// per byte: many tokens) or 16 (one load, an 8-byte store, half the work per
// lane on the dependent path: few tokens).  Every thread first issues its
// loads of the piece; each warp reads the token's destination rows itself
// (one lane per rank, ballot) while they are in flight.  Then per round each
// group of kLanes lanes reduces its block's amax by shuffles, forms the scale
// and the codes, and stores the code vector (and, its first lane, the scale)
// to every destination.
template <bool kExpanded, int kLanes, bool kSelf, int kMW = kMetaWarps>
__device__ __forceinline__ void dispatch_fp8_item(const DispatchParams& p, int64_t it, int gtid, int lane,
                                                  int group_warps, bool& cap_bad, bool signal = false) {
    constexpr int kVec = 128 / kLanes / 8;                     // 16-byte input vectors per lane per block
    constexpr int kBlocksPerWarp = 32 / kLanes;
    const int blocks_per_round = kBlocksPerWarp * group_warps;
    const int t = static_cast<int>(it / p.chunks);
    const int c = static_cast<int>(it - static_cast<int64_t>(t) * p.chunks);
    const int warp_g = gtid >> 5;
    const int grp = lane / kLanes;
    const int sub = lane % kLanes;
    const int nb = p.H / 128;
    const int b_begin = c * p.chunk_blocks;
    const int b_end = min(nb, b_begin + p.chunk_blocks);
    const int64_t xrow_off = static_cast<int64_t>(t) * p.H * 2, x_bytes = static_cast<int64_t>(p.T) * p.H * 2;
    const uint8_t* xrow = p.x + xrow_off;
    uint4 v[kFp8Rounds][kVec];
#pragma unroll
    for (int q = 0; q < kFp8Rounds; ++q) {
        const int b = b_begin + q * blocks_per_round + kBlocksPerWarp * warp_g + grp;
        const int64_t so = static_cast<int64_t>(b) * 256 + sub * (16 * kVec);
        const uint8_t* src = xrow + so;
#pragma unroll
        for (int u = 0; u < kVec; ++u)
            v[q][u] = (b < b_end && EP_IN_BYTES(xrow_off + so + 16 * u, 16, x_bytes))
                          ? ld_stream_v4(src + 16 * u)
                          : make_uint4(0, 0, 0, 0);
    }
    const int n_dst = kExpanded ? p.K : p.R;
    const int64_t drow0 = static_cast<int64_t>(t) * n_dst, n_drow = static_cast<int64_t>(p.T) * n_dst;
    const int32_t* drow = (kExpanded ? p.expanded_row : p.dst_row) + drow0;
    int d0, d1;
    int64_t me_l = -1;   // self-routed: the token's entries, for the receive metadata
    float mw_l = 0.0f;
    if constexpr (kSelf) {
        if (EP_SELF_EARLY_META && static_cast<unsigned>(self_meta_part(p, c, warp_g, group_warps)) < 2u)
            load_token_entries(p, t, lane, me_l, mw_l);
        d0 = self_route_layout<false>(p, t, c, self_smem());   // R <= 32
        d1 = -1;
    } else {
        if (signal) wait_rows_ready(p, t);   // x is already in flight
        d0 = (lane < n_dst && EP_IN(drow0 + lane, n_drow)) ? drow[lane] : -1;
        d1 = (32 + lane < n_dst && EP_IN(drow0 + 32 + lane, n_drow)) ? drow[32 + lane] : -1;   // ranks 32..63
        (void)EP_ROW_OK(d0);
        (void)EP_ROW_OK(d1);
    }
    const int64_t rx_bytes = p.capacity * p.H;   // FP8 codes: one byte per channel
    const int64_t sf_n = p.sf_col_major ? static_cast<int64_t>(nb) * p.sf_stride : p.capacity * nb;
    if (kSelf) {
        const int part = self_meta_part(p, c, warp_g, group_warps);
        if (part >= 0) {
            if (!EP_SELF_EARLY_META && part < 2) load_token_entries(p, t, lane, me_l, mw_l);
            write_metadata_part(p, t, lane, d0, me_l, mw_l, part);
        }
    } else if (c == 0 && (kExpanded ? warp_g == 1 : (warp_g >= 1 && warp_g <= kMW))) {
        if (kExpanded) {
            write_expanded_metadata(p, t, lane);
        } else {
            CtaWork all;
            all.first = 0;
            all.count = 0;
            all.stride = 1;
            all.lo = INT32_MIN;
            all.hi = INT32_MAX;
            all.balanced = 0;
            // one array per warp (kMW == 3), or all on warp 1
            write_metadata(p, t, lane, all, kMW == 3 ? warp_g - 1 : -1);
        }
    }
    // Many tokens (kLanes 8): codes and scales of every round first, then one
    // pass over the destinations stores all of them (one shuffle and one row
    // address per destination instead of one per round).  Few tokens (kLanes
    // 16): each round is stored as soon as it is cast, which keeps the first
    // stores early on the short, latency-bound grid.
    constexpr bool kMerged = kLanes == 8;
    const int b0 = b_begin + kBlocksPerWarp * warp_g + grp;   // this lane's block in round 0
    uint32_t code[kFp8Rounds][2 * kVec];
    float sfq[kFp8Rounds];
    auto warp_has_round = [&](int q) { return b_begin + q * blocks_per_round + kBlocksPerWarp * warp_g < b_end; };
    auto cast_round = [&](int q) {
        sfq[q] = 1.0f;
#pragma unroll
        for (int e = 0; e < 2 * kVec; ++e) code[q][e] = 0u;
        float f[8 * kVec];
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            const uint32_t w[4] = {v[q][u].x, v[q][u].y, v[q][u].z, v[q][u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[8 * u + 2 * e] = __uint_as_float(w[e] << 16);
                f[8 * u + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 8 * kVec; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
        for (int o = kLanes / 2; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        float mult = 0.0f;
        if (amax > 0.0f) {
            sfq[q] = __fdiv_rn(amax, 448.0f);
            mult = __fdiv_rn(448.0f, amax);
        }
        if (kMerged) {   // packed products: fewer instructions on the issue-heavy many-token grid
            uint64_t mm;
            asm("mov.b64 %0, {%1, %1};" : "=l"(mm) : "f"(mult));
#pragma unroll
            for (int e = 0; e < 2 * kVec; ++e) {
                const float2 lo = mul2_rn(f[4 * e], f[4 * e + 1], mm);
                const float2 hi = mul2_rn(f[4 * e + 2], f[4 * e + 3], mm);
                code[q][e] = pack_e4m3x4(lo.x, lo.y, hi.x, hi.y);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 2 * kVec; ++e)
                code[q][e] = pack_e4m3x4(__fmul_rn(f[4 * e], mult), __fmul_rn(f[4 * e + 1], mult),
                                         __fmul_rn(f[4 * e + 2], mult), __fmul_rn(f[4 * e + 3], mult));
        }
    };
    const int sub_col = sub * (8 * kVec);
    // stores rounds [q_lo, q_hi) to every destination
    auto store_rounds = [&](int q_lo, int q_hi) {
        for (int rb = 0; rb < n_dst; rb += 32) {
            const int d = rb == 0    ? d0
                          : rb == 32 ? d1
                                     : ((rb + lane < n_dst && EP_IN(drow0 + rb + lane, n_drow)) ? drow[rb + lane] : -1);
            if (rb >= 64) (void)EP_ROW_OK(d);
            if (d >= p.capacity && c == 0 && q_lo == 0) cap_bad = true;
            unsigned m = __ballot_sync(0xffffffffu, d >= 0 && d < p.capacity);
            while (m) {
                const int sl = __ffs(m) - 1;
                m &= m - 1;
                const int64_t dd = __shfl_sync(0xffffffffu, d, sl);
                uint8_t* row = p.recv_x + dd * p.H + sub_col;
#pragma unroll
                for (int q = 0; q < kFp8Rounds; ++q) {
                    const int b = b0 + q * blocks_per_round;
                    if (q >= q_lo && q < q_hi && b < b_end &&
                        EP_IN_BYTES(dd * p.H + sub_col + static_cast<int64_t>(b) * 128, 8 * kVec, rx_bytes)) {
                        uint8_t* dst = row + static_cast<int64_t>(b) * 128;
                        if (kVec == 2)
                            st_v4(dst, make_uint4(code[q][0], code[q][1], code[q][2 % (2 * kVec)],
                                                  code[q][3 % (2 * kVec)]));
                        else
                            *reinterpret_cast<uint2*>(dst) = make_uint2(code[q][0], code[q][1]);
                        if (sub == 0 && p.recv_sf) {
                            const int64_t si =
                                p.sf_col_major ? static_cast<int64_t>(b) * p.sf_stride + dd : dd * nb + b;
                            if (EP_IN(si, sf_n)) p.recv_sf[si] = sfq[q];
                        }
                    }
                }
            }
        }
    };
    if constexpr (kMerged && EP_DISPATCH_FP8_HOISTED) {
#pragma unroll
        for (int q = 0; q < kFp8Rounds; ++q)
            if (warp_has_round(q)) cast_round(q);   // warp-uniform
        // Every per-lane offset, predicate and base pointer is formed once,
        // outside the destination loop, which then costs one row address,
        // two predicated 16-byte code stores and, on a block's first lane,
        // two predicated scale stores per destination.
        static_assert(kFp8Rounds == 2 && kVec == 2, "the hoisted store pass handles two rounds of 16-byte codes");
        const int bq0 = b0, bq1 = b0 + blocks_per_round;
        const bool ok0 = bq0 < b_end, ok1 = bq1 < b_end;
        const int64_t co0 = static_cast<int64_t>(bq0) * 128 + sub_col;
        const int64_t co1 = static_cast<int64_t>(bq1) * 128 + sub_col;
        uint8_t* const rx = p.recv_x;
        float* const rsf = p.recv_sf;
        const int64_t H = p.H, cap = p.capacity;
        const bool sf_lane = sub == 0 && rsf != nullptr;
        const bool col = p.sf_col_major != 0;
        const int64_t sfs = col ? 1 : nb;                                   // scale index = dd * sfs + so_q
        const int64_t so0 = col ? static_cast<int64_t>(bq0) * p.sf_stride : bq0;
        const int64_t so1 = col ? static_cast<int64_t>(bq1) * p.sf_stride : bq1;
        const uint4 c0 = make_uint4(code[0][0], code[0][1], code[0][2], code[0][3]);
        const uint4 c1 = make_uint4(code[1][0], code[1][1], code[1][2], code[1][3]);
#if EP_DISPATCH_FP8_L2
        const uint64_t code_pol = l2_policy_evict_first();
        if (p.prefetch_evict_last) {   // this lane's x vectors are read: lines they start back to normal
#pragma unroll
            for (int q = 0; q < kFp8Rounds; ++q) {
                const int b = b_begin + q * blocks_per_round + kBlocksPerWarp * warp_g + grp;
                const uint8_t* a = xrow + static_cast<int64_t>(b) * 256 + sub * (16 * kVec);
                if (b < b_end && (reinterpret_cast<uintptr_t>(a) & 127u) == 0 &&
                    xrow_off + static_cast<int64_t>(b) * 256 + sub * (16 * kVec) + 128 <= x_bytes)
                    l2_priority_normal(a);
            }
        }
#endif
        const float s0 = sfq[0], s1 = sfq[1];
        for (int rb = 0; rb < n_dst; rb += 32) {
            const int d = rb == 0    ? d0
                          : rb == 32 ? d1
                                     : ((rb + lane < n_dst && EP_IN(drow0 + rb + lane, n_drow)) ? drow[rb + lane] : -1);
            if (rb >= 64) (void)EP_ROW_OK(d);
            if (d >= cap && c == 0) cap_bad = true;
            unsigned m = __ballot_sync(0xffffffffu, d >= 0 && d < cap);
            while (m) {
                const int sl = __ffs(m) - 1;
                m &= m - 1;
                const int64_t dd = __shfl_sync(0xffffffffu, d, sl);
                uint8_t* row = rx + dd * H;
#if EP_DISPATCH_FP8_L2
                if (ok0 && EP_IN_BYTES(dd * H + co0, 16, rx_bytes)) st_v4_hint(row + co0, c0, code_pol);
                if (ok1 && EP_IN_BYTES(dd * H + co1, 16, rx_bytes)) st_v4_hint(row + co1, c1, code_pol);
#else
                if (ok0 && EP_IN_BYTES(dd * H + co0, 16, rx_bytes)) *reinterpret_cast<uint4*>(row + co0) = c0;
                if (ok1 && EP_IN_BYTES(dd * H + co1, 16, rx_bytes)) *reinterpret_cast<uint4*>(row + co1) = c1;
#endif
                if (sf_lane) {
                    float* srow = rsf + dd * sfs;
                    if (ok0 && EP_IN(dd * sfs + so0, sf_n)) srow[so0] = s0;
                    if (ok1 && EP_IN(dd * sfs + so1, sf_n)) srow[so1] = s1;
                }
            }
        }
    } else if constexpr (kMerged) {
#pragma unroll
        for (int q = 0; q < kFp8Rounds; ++q)
            if (warp_has_round(q)) cast_round(q);   // warp-uniform
        store_rounds(0, kFp8Rounds);
    } else {
#pragma unroll
        for (int q = 0; q < kFp8Rounds; ++q) {
            if (!warp_has_round(q)) break;   // warp-uniform
            cast_round(q);
            store_rounds(q, q + 1);
        }
    }
}

// kGroups == 1: one CTA per item.  kGroups > 1 (SM-limited mode): several
// independent groups per CTA, each looping over items with a stride.
// The many-token rank-row instantiation runs 5 CTAs per SM (more loads in
// flight; 4 for the few-token and expanded ones, which the cap would slow or
// spill).
template <bool kExpanded, int kGroups, int kLanes, bool kSelf = false>
__global__ void __launch_bounds__(kFp8Threads * kGroups,
                                  kGroups > 1 ? 1
                                  : (kLanes == 8 && !kExpanded) ? EP_DISPATCH_FP8_WIDE_MIN_BLOCKS
                                                                : EP_DISPATCH_FP8_MIN_BLOCKS)
    dispatch_fp8_kernel(const DispatchParams p) {
    // one CTA per item: blockDim.x / 32 warps (up to 8, as many as the
    // piece's blocks need); SM-limited groups: 8 warps each
    const int gtid = kGroups == 1 ? static_cast<int>(threadIdx.x) : static_cast<int>(threadIdx.x) % kFp8Threads;
    const int lane = threadIdx.x & 31;
    bool cap_bad = false;
    if (kSelf && blockIdx.x >= gridDim.x - kSelfLayoutCtas) {   // the layout's counts and offsets
        pdl_wait();
        self_route_layout<true>(p, 0, static_cast<int>(gridDim.x - 1 - blockIdx.x), self_smem());
        return;
    }
    if (kGroups == 1) prefetch_x<true>(p);
    // with the rows-ready signal (first wave) only dst_row waits (see the
    // bf16 kernel)
    const bool signal_call = kGroups == 1 && !kSelf && !kExpanded && p.rows_ready != nullptr;
    const bool signal = signal_call && static_cast<int>(blockIdx.x) < p.rows_first_wave;
    if (!signal) pdl_wait();   // before any load: the previous kernel may write x
    if (kGroups == 1) {
        dispatch_fp8_item<kExpanded, kLanes, kSelf>(p, blockIdx.x, gtid, lane, static_cast<int>(blockDim.x) / 32,
                                                    cap_bad, signal);
        if (signal_call && blockIdx.x == gridDim.x - 1) clear_rows_slots(p);
    } else {
        const int64_t n_items = static_cast<int64_t>(p.T) * p.chunks;
        const int group = static_cast<int>(threadIdx.x) / kFp8Threads;
        for (int64_t it = static_cast<int64_t>(blockIdx.x) * kGroups + group; it < n_items;
             it += static_cast<int64_t>(gridDim.x) * kGroups)
            dispatch_fp8_item<kExpanded, kLanes, false, 1>(p, it, gtid, lane, kFp8Threads / 32, cap_bad);
    }
    if ((gtid >> 5) == 0 && __any_sync(0xffffffffu, cap_bad) && lane == 0) atomicOr(p.status, EP_ERR_CAPACITY);
}

// Bulk-copy path: the default alternative (EP_DISPATCH_IMPL=0) and the
// SM-limited mode (num_sms > 0, one CTA per SM with a deeper ring).
template <int kStages, int kStoreDepth>
cudaError_t launch_dispatch_bulk_t(DispatchParams p, int max_ctas, cudaStream_t stream) {
    const DeviceInfo& di = device_info();
    const uint32_t row_bytes = static_cast<uint32_t>(p.H) * 2u;
    int chunks = static_cast<int>((row_bytes + EP_DISPATCH_PIECE_MAX - 1) / EP_DISPATCH_PIECE_MAX);
    const int want_items = 2 * di.num_sms;
    if (p.T > 0 && static_cast<int64_t>(p.T) * chunks < want_items) {
        const int more = (want_items + p.T - 1) / p.T;
        const int max_chunks = static_cast<int>(row_bytes / 1024u) > 0 ? static_cast<int>(row_bytes / 1024u) : 1;
        chunks = more < max_chunks ? more : max_chunks;
        if (chunks < 1) chunks = 1;
    }
    uint32_t chunk_bytes = (row_bytes + chunks - 1) / chunks;
    chunk_bytes = (chunk_bytes + 15u) / 16u * 16u;
    chunks = static_cast<int>((row_bytes + chunk_bytes - 1) / chunk_bytes);
    p.chunks = chunks;
    p.chunk_bytes = chunk_bytes;
    const size_t smem = 128 + static_cast<size_t>(kStages) * chunk_bytes;

    static thread_local int configured_device = -1;
    static thread_local int blocks_per_sm = 1;
    static thread_local size_t configured_smem = 0;
    if (configured_device != di.device || configured_smem != smem) {
        cudaError_t e = cudaFuncSetAttribute(dispatch_bf16_kernel<kStages, kStoreDepth>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, dispatch_bf16_kernel<kStages, kStoreDepth>,
                                                          kBf16Threads, smem);
        if (e != cudaSuccess) return e;
        blocks_per_sm = nb > 0 ? nb : 1;
        configured_device = di.device;
        configured_smem = smem;
    }
    const int64_t num_items = static_cast<int64_t>(p.T) * chunks;
    int64_t grid = static_cast<int64_t>(di.num_sms) * blocks_per_sm;
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    if (grid > num_items) grid = num_items;
    if (grid < 1) return cudaSuccess;
    return launch_pdl(dispatch_bf16_kernel<kStages, kStoreDepth>, dim3(static_cast<unsigned>(grid)),
                      dim3(kBf16Threads), smem, stream, p);
}

}  // namespace

cudaError_t launch_dispatch_bf16(DispatchParams p, cudaStream_t stream) {
    const DeviceInfo& di = device_info();
    const uint32_t row_bytes = static_cast<uint32_t>(p.H) * 2u;
    if (p.num_sms > 0 && p.expanded_row == nullptr) {
        // SM-limited rank-row dispatch: the bulk-copy kernel with the deep
        // ring; at most num_sms CTAs (one per SM for rows of 6 KB or more)
        const int n = p.num_sms < di.num_sms ? p.num_sms : di.num_sms;
        return launch_dispatch_bulk_t<kSmBulkStages, kSmBulkStoreDepth>(p, n, stream);
    }
    if (EP_DISPATCH_IMPL == 1 || p.expanded_row != nullptr) {
        // register path (the expanded mode always takes it): one CTA per (token, piece of <= 16 KB); more pieces for few tokens
        int chunks = static_cast<int>((row_bytes + 16383u) / 16384u);
        const int want_items = 4 * di.num_sms;
        if (p.T > 0 && static_cast<int64_t>(p.T) * chunks < want_items) {
            // a CTA that derives its rows itself (self_route) pays that
            // latency once per wave: keep it to one wave of 4 CTAs per SM
            // (the layout CTAs included)
            const int more = p.self_route ? (di.num_sms * kSelfRegBlocks - kSelfLayoutCtas) / p.T
                                          : (want_items + p.T - 1) / p.T;
            const int max_chunks = static_cast<int>(row_bytes / 1024u) > 0 ? static_cast<int>(row_bytes / 1024u) : 1;
            chunks = more < max_chunks ? more : max_chunks;
            if (chunks < 1) chunks = 1;
        }
        uint32_t cb = (row_bytes + chunks - 1) / chunks;
        cb = (cb + 15u) / 16u * 16u;
        p.chunks = static_cast<int>((row_bytes + cb - 1) / cb);
        p.chunk_bytes = cb;
        const int64_t items = static_cast<int64_t>(p.T) * p.chunks;
        if (items < 1) return cudaSuccess;
        const int num_sms = p.num_sms > 0 ? (p.num_sms < di.num_sms ? p.num_sms : di.num_sms) : 0;
        if (num_sms > 0) {   // only the expanded mode reaches here (rank rows took the bulk path)
            int64_t g = (items + kSmGroups - 1) / kSmGroups;
            if (g > num_sms) g = num_sms;
            const dim3 grid(static_cast<unsigned>(g)), block(kRegThreads * kSmGroups);
            return launch_pdl(dispatch_bf16_regs_kernel<true, kSmGroups>, grid, block, 0, stream, p);
        }
        // self routing: kSelfLayoutCtas more CTAs, which write the layout's counts and offsets
        const dim3 grid(static_cast<unsigned>(items + (p.self_route ? kSelfLayoutCtas : 0))), block(kRegThreads);
        p.prefetch_ctas = di.num_sms * 6;   // the first wave (6 CTAs per SM)
        p.rows_first_wave = p.prefetch_ctas;
        // the first wave prefetches the pieces of every generation while they
        // fit the L2 budget (all of x on DeepSeek-V3-sized inputs)
        {
            const int64_t budget_items = static_cast<int64_t>(EP_DISPATCH_PREFETCH_L2_BYTES) / cb;
            const int64_t n_pf = items < budget_items ? items : budget_items;
            int64_t gens = n_pf / p.prefetch_ctas;
            if (gens < 1) gens = 1;
            if (gens > EP_DISPATCH_PREFETCH_MAX_GENS) gens = EP_DISPATCH_PREFETCH_MAX_GENS;
            p.prefetch_items = static_cast<int>(gens);
            p.prefetch_evict_last = EP_DISPATCH_PREFETCH_EVICT_LAST;
        }
        if (p.expanded_row) return launch_pdl(dispatch_bf16_regs_kernel<true, 1>, grid, block, 0, stream, p);
        if (p.self_route) return launch_pdl(dispatch_bf16_regs_kernel<false, 1, true>, grid, block, 0, stream, p);
        return launch_pdl(dispatch_bf16_regs_kernel<false, 1>, grid, block, 0, stream, p);
    }
    return launch_dispatch_bulk_t<kBulkStages, kBulkStoreDepth>(p, 0, stream);
}

template <int kLanes>
cudaError_t launch_dispatch_fp8_t(DispatchParams p, int num_sms, cudaStream_t stream) {
    const int64_t items = static_cast<int64_t>(p.T) * p.chunks;
    if (num_sms > 0) {
        int64_t g = (items + kSmGroups - 1) / kSmGroups;
        if (g > num_sms) g = num_sms;
        const dim3 grid(static_cast<unsigned>(g)), block(kFp8Threads * kSmGroups);
        if (p.expanded_row) return launch_pdl(dispatch_fp8_kernel<true, kSmGroups, kLanes>, grid, block, 0, stream, p);
        return launch_pdl(dispatch_fp8_kernel<false, kSmGroups, kLanes>, grid, block, 0, stream, p);
    }
    // Many tokens: as many warps per CTA as the piece's blocks need (a warp
    // casts 4 blocks per round), so a 56-block row (H = 7168) runs 7 warps
    // with no idle lanes and fits 6 CTAs per SM instead of 5.
    int warps = kFp8Threads / 32;
    if (kLanes == 8 && EP_DISPATCH_FP8_FIT_WARPS) {
        warps = (p.chunk_blocks + kFp8Rounds * 4 - 1) / (kFp8Rounds * 4);
        if (warps > kFp8Threads / 32) warps = kFp8Threads / 32;
        if (warps < 1 + kMetaWarps) warps = 1 + kMetaWarps;   // warps 1 .. kMetaWarps write the metadata
    }
    // self routing (few tokens, the 16-lane mode): kSelfLayoutCtas more CTAs,
    // which write the layout's counts and offsets
    const bool self = kLanes == 16 && p.self_route && !p.expanded_row;
    const dim3 grid(static_cast<unsigned>(items + (self ? kSelfLayoutCtas : 0))), block(32 * warps);
    auto kernel = p.expanded_row ? dispatch_fp8_kernel<true, 1, kLanes>
                  : (kLanes == 16 && p.self_route) ? dispatch_fp8_kernel<false, 1, 16, true>
                                                   : dispatch_fp8_kernel<false, 1, kLanes>;
    // CTAs resident per SM at this size: the first wave, which prefetches
    static thread_local int occ_device = -1, occ_threads = 0, occ_kind = -1, occ_ctas = 1;
    const int dev = device_info().device;
    const int kind = p.expanded_row ? 1 : p.self_route ? 2 : 0;
    if (occ_device != dev || occ_threads != 32 * warps || occ_kind != kind) {
        int nb_sm = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb_sm, kernel, 32 * warps, 0);
        if (e != cudaSuccess) return e;
        occ_ctas = nb_sm > 0 ? nb_sm : 1;
        occ_device = dev;
        occ_threads = 32 * warps;
        occ_kind = kind;
    }
    p.prefetch_ctas = device_info().num_sms * occ_ctas;
    p.rows_first_wave = p.prefetch_ctas;
    p.prefetch_items = EP_DISPATCH_PREFETCH;
    p.prefetch_evict_last = 0;
    if (EP_DISPATCH_FP8_L2 && !self && !p.expanded_row) {
        // the bf16 path's L2 policy: every generation of pieces within the
        // budget, prefetched evict-last by the first wave
        const int64_t piece = static_cast<int64_t>(p.chunk_blocks) * 256;
        const int64_t n_items = static_cast<int64_t>(p.T) * p.chunks;
        const int64_t budget_items = static_cast<int64_t>(EP_DISPATCH_PREFETCH_L2_BYTES) / piece;
        int64_t gens = (n_items < budget_items ? n_items : budget_items) / p.prefetch_ctas;
        if (gens < 1) gens = 1;
        if (gens > EP_DISPATCH_PREFETCH_MAX_GENS) gens = EP_DISPATCH_PREFETCH_MAX_GENS;
        p.prefetch_items = static_cast<int>(gens);
        p.prefetch_evict_last = 1;
    }
    return launch_pdl(kernel, grid, block, 0, stream, p);
}

bool dispatch_reads_rows_signal(bool fp8) {
    return fp8 ? (EP_ROWS_SIGNAL & 2) != 0 : ((EP_ROWS_SIGNAL & 1) != 0 && EP_DISPATCH_IMPL == 1);
}

cudaError_t launch_dispatch_fp8(DispatchParams p, cudaStream_t stream) {
    const DeviceInfo& di = device_info();
    const int nb = p.H / 128;
    // Many tokens: 8 lanes per block (fewer instructions per byte); few tokens
    // (fewer than 8 per SM): 16 lanes per block (shorter dependent path).
    const bool wide = static_cast<int64_t>(p.T) >= 8 * static_cast<int64_t>(di.num_sms);
    const int blocks_per_round = (wide ? 4 : 2) * (kFp8Threads / 32);
    // One CTA per (token, piece); pieces of up to kFp8Rounds rounds of blocks
    // (at most EP_DISPATCH_FP8_PIECE_BLOCKS), split further when there are few tokens.
    int piece_max = kFp8Rounds * blocks_per_round;
    if (piece_max > EP_DISPATCH_FP8_PIECE_BLOCKS) piece_max = EP_DISPATCH_FP8_PIECE_BLOCKS;
    int chunks = (nb + piece_max - 1) / piece_max;
    const int want_items = 4 * di.num_sms;
    if (p.T > 0 && static_cast<int64_t>(p.T) * chunks < want_items) {
        // a CTA that derives its rows itself (self_route) pays that latency
        // once per wave: keep it to one wave of 4 CTAs per SM, the layout
        // CTAs included
        const int more = p.self_route ? (want_items - kSelfLayoutCtas) / p.T : (want_items + p.T - 1) / p.T;
        const int max_chunks = (nb + blocks_per_round / 8 - 1) / (blocks_per_round / 8);   // >= one warp's blocks per piece
        chunks = more < max_chunks ? more : max_chunks;
        if (chunks < 1) chunks = 1;
    }
    int chunk_blocks = (nb + chunks - 1) / chunks;
    chunks = (nb + chunk_blocks - 1) / chunk_blocks;
    p.chunks = chunks;
    p.chunk_blocks = chunk_blocks;
    const int64_t items = static_cast<int64_t>(p.T) * chunks;
    if (items < 1) return cudaSuccess;
    const int num_sms = p.num_sms > 0 ? (p.num_sms < di.num_sms ? p.num_sms : di.num_sms) : 0;
    return wide ? launch_dispatch_fp8_t<8>(p, num_sms, stream) : launch_dispatch_fp8_t<16>(p, num_sms, stream);
}

}  // namespace epg
