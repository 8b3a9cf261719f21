// Combine: gather each token's expert-output rows back from the receive rows
// and reduce them into token order ("DeepEP Symmetric Memory" section 9.2,
// combine(x, handle, topk_weights) -> combined_x):
//   out[t] = bf16_rne( sum over ranks r holding t of c(t,r) * y[dst_row[t,r]] )
// with fp32 accumulation; c = 1 unweighted, else the sum of t's top-k weights
// whose expert lives on r.
//
// One CTA of 128 threads per (token, piece of the row).  Warp 0 compacts the
// token's receive rows (ascending rank) and coefficients into shared memory;
// then every thread owns 16-byte vectors of the piece and issues the loads of
// up to 4 source rows back to back (read-only, no L1 allocation) before
// accumulating (64 bytes of reads in flight per thread, 12 CTAs per SM).  The
// reduced vector is rounded to bf16 and stored once.  HBM-bound: reads are
// ~n(t) times the writes.
//
// SM-limited mode (num_sms > 0): CTAs of 8 groups of 128 threads, one per SM,
// each group looping over whole-row items (pieces only when there are fewer
// rows than groups) with 8 source rows of loads in flight per thread (same
// order and arithmetic, so results are bit-identical).  Shared-memory rings
// fed by bulk copies (per-row slots, or per-item stages with one to four
// producer warps) measured 30% to 2.8x slower: their handshakes cost more than
// register loads.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace epg {
namespace {

// Compile-time tuning (defaults are the measured best on GB300).
#ifndef EP_COMBINE_THREADS
#define EP_COMBINE_THREADS 128       // threads per CTA
#endif
#ifndef EP_COMBINE_MIN_BLOCKS
#define EP_COMBINE_MIN_BLOCKS 12     // __launch_bounds__ minimum resident CTAs per SM (<= 40 registers)
#endif
constexpr int kThreads = EP_COMBINE_THREADS;
#ifndef EP_COMBINE_PREFETCH_ROWS
#define EP_COMBINE_PREFETCH_ROWS 1   // warp 0 asks L2 for the row pieces past the first batch
#endif
#ifndef EP_COMBINE_BATCH
#define EP_COMBINE_BATCH 4
#endif
// Many tokens: 16-byte vectors per thread in a piece.  Rank rows (~5 per
// token on DS-V3) take 2; expanded rows (K = 8 per token, two batches of
// loads per vector) take 1, so that a CTA waits on fewer round trips
// (DS-V3 expanded combine 78.1 -> 75.8 us; rank rows with 1: 53.6 -> 54.7 us).
#ifndef EP_COMBINE_VECS
#define EP_COMBINE_VECS 2
#endif
#ifndef EP_COMBINE_VECS_EXPANDED
#define EP_COMBINE_VECS_EXPANDED 1
#endif
constexpr int kCombineVecs = EP_COMBINE_VECS;
constexpr int kCombineVecsExpanded = EP_COMBINE_VECS_EXPANDED;
constexpr int kBatch = EP_COMBINE_BATCH;
#ifndef EP_COMBINE_SM_BATCH
#define EP_COMBINE_SM_BATCH 8        // SM-limited mode: rows of loads in flight per thread
#endif
#ifndef EP_COMBINE_FEW_BATCH
#define EP_COMBINE_FEW_BATCH 8       // few tokens: rows of loads in flight per thread
#endif
#ifndef EP_COMBINE_FEW_MIN_BLOCKS
#define EP_COMBINE_FEW_MIN_BLOCKS 6  // few tokens: minimum resident CTAs per SM (78 registers, unspilled)
#endif

// SM-limited mode: CTAs of kSmGroups x kThreads threads, one per SM, each
// group looping over (token, piece) items.
constexpr int kSmGroups = 8;

// One (token, piece) item, by one group of kThreads threads.  kExpanded: the
// token's source rows are its expanded rows (one per valid top-k slot,
// coefficient = that slot's weight) instead of one row per rank.  kB: source
// rows of loads in flight per thread.
// Pairs of fp32 in one 64-bit register, added or fused-multiply-added by the
// packed fp32x2 instructions: each element is rounded as by the scalar
// instruction, so sums are bit-identical to scalar code, with half the adds.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo_bits, uint32_t hi_bits) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}

// Asks L2 for `bytes` (a multiple of 16) at the 16-byte aligned `ptr`.
__device__ __forceinline__ void prefetch_piece_l2(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

template <bool kWeighted, bool kExpanded, int kGroups, int kB>
__device__ __forceinline__ void combine_item(const CombineParams& p, int64_t it, int group, int gtid,
                                             int* s_rows, float* s_coef, int* s_n) {
    const int t = static_cast<int>(it / p.chunks);
    const int c = static_cast<int>(it - static_cast<int64_t>(t) * p.chunks);
    if (gtid < 32) {
        const int lane = gtid;
        int64_t e_l = -1;
        float w_l = 0.0f;
        if (kWeighted && lane < p.K && EP_IN(static_cast<int64_t>(t) * p.K + lane, static_cast<int64_t>(p.T) * p.K)) {
            if (!kExpanded) e_l = p.topk_idx[static_cast<int64_t>(t) * p.K + lane];
            w_l = p.topk_weights[static_cast<int64_t>(t) * p.K + lane];
        }
        int n = 0;
        bool cap_bad = false;
        const int n_src = kExpanded ? p.K : p.R;
        const int64_t srow0 = static_cast<int64_t>(t) * n_src, n_srow = static_cast<int64_t>(p.T) * n_src;
        const int32_t* srow = (kExpanded ? p.expanded_row : p.dst_row) + srow0;
        for (int rb = 0; rb < n_src; rb += 32) {
            const int r = rb + lane;
            const int d = (r < n_src && EP_IN(srow0 + r, n_srow)) ? srow[r] : -1;
            (void)EP_ROW_OK(d);
            const bool ok = d >= 0 && d < p.num_y_rows;
            if (d >= p.num_y_rows) cap_bad = true;
            float coef = 1.0f;
            if (kExpanded) {
                if (kWeighted) coef = w_l;   // lane r holds slot r's weight (K <= 32)
            } else if (kWeighted) {
                coef = 0.0f;
                for (int k = 0; k < p.K; ++k) {
                    const int64_t e = __shfl_sync(0xffffffffu, e_l, k);
                    const float w = __shfl_sync(0xffffffffu, w_l, k);
                    if (e >= 0 && e < p.E && static_cast<int>(e) / p.experts_per_rank == r) coef += w;
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, ok);
            const int pos = n + __popc(m & ((1u << lane) - 1u));
#if EP_COMBINE_PREFETCH_ROWS
            // rank rows past the first batch: this item's piece of the row
            // into L2 now, so that the second batch of loads after the
            // barrier finds it there (the first batch's loads are issued right
            // away anyway).  Not on the expanded rows, where it measured slower.
            if (kGroups == 1 && !kExpanded && ok && pos >= kB) {
                const int64_t rb_bytes = static_cast<int64_t>(p.H) * 2;
                const int64_t off = static_cast<int64_t>(c) * p.chunk_vecs * 16;
                const int64_t len = min(static_cast<int64_t>(p.chunk_vecs) * 16, rb_bytes - off);
                if (len > 0 && EP_IN_BYTES(static_cast<int64_t>(d) * rb_bytes + off, len, p.num_y_rows * rb_bytes))
                    prefetch_piece_l2(p.y + static_cast<int64_t>(d) * rb_bytes + off, static_cast<uint32_t>(len));
            }
#endif
            // A layout from ep_get_layout has at most K <= 32 ranks per token;
            // a foreign dst_row with more is cut off and flagged.
            if (ok && pos < EP_MAX_TOPK) {
                s_rows[pos] = d;
                s_coef[pos] = coef;
            }
            n += __popc(m);
        }
        if (n > EP_MAX_TOPK) {
            if (lane == 0) atomicOr(p.status, EP_ERR_INVALID_INDEX);
            n = EP_MAX_TOPK;
        }
        if (lane == 0) *s_n = n;
        if (__any_sync(0xffffffffu, cap_bad) && lane == 0 && c == 0) atomicOr(p.status, EP_ERR_CAPACITY);
    }
    if (kGroups > 1)
        named_barrier(1 + group, kThreads);
    else
        __syncthreads();

    const int n = *s_n;
    const int n_vec = p.H / 8;
    const int v_begin = c * p.chunk_vecs;
    const int v_end = min(n_vec, v_begin + p.chunk_vecs);
    const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
    const int64_t y_bytes = p.num_y_rows * row_bytes, out_bytes = static_cast<int64_t>(p.T) * row_bytes;
    for (int v = v_begin + gtid; v < v_end; v += kThreads) {
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};   // channel pairs (2q, 2q + 1), +0.0f each
        const int64_t off = static_cast<int64_t>(v) * 16;
        for (int m0 = 0; m0 < n; m0 += kB) {
            uint4 buf[kB];
#pragma unroll
            for (int j = 0; j < kB; ++j)
                if (m0 + j < n) {
                    const int64_t yo = static_cast<int64_t>(s_rows[m0 + j]) * row_bytes + off;
                    buf[j] = EP_IN_BYTES(yo, 16, y_bytes) ? ld_stream_v4(p.y + yo) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                if (m0 + j < n) {
                    const uint32_t w[4] = {buf[j].x, buf[j].y, buf[j].z, buf[j].w};
                    if (kWeighted) {
                        const uint32_t cb = __float_as_uint(s_coef[m0 + j]);
                        const uint64_t cf2 = f2_pack(cb, cb);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            acc[q] = f2_fma(cf2, f2_pack(w[q] << 16, w[q] & 0xffff0000u), acc[q]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[q] = f2_add(acc[q], f2_pack(w[q] << 16, w[q] & 0xffff0000u));
                    }
                }
            }
        }
        uint4 o;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 a = f2_unpack(acc[q]);
            const __nv_bfloat162 h = __floats2bfloat162_rn(a.x, a.y);
            ow[q] = *reinterpret_cast<const uint32_t*>(&h);
        }
        if (EP_IN_BYTES(static_cast<int64_t>(t) * row_bytes + off, 16, out_bytes))
            st_v4(p.out + static_cast<int64_t>(t) * row_bytes + off, o);
    }
}

// kGroups == 1: one CTA per item.  kGroups > 1 (SM-limited mode): several
// groups per CTA, each looping over items with a stride and synchronising on
// its own named barrier.  kB > kBatch with kGroups == 1: the few-token grid,
// where one round trip for all of a token's rows matters more than occupancy.
template <bool kWeighted, bool kExpanded, int kGroups, int kB>
__global__ void __launch_bounds__(kThreads * kGroups,
                                  kGroups > 1 ? 1 : (kB > kBatch ? EP_COMBINE_FEW_MIN_BLOCKS : EP_COMBINE_MIN_BLOCKS))
    combine_kernel(const CombineParams p) {
    __shared__ int s_rows_all[kGroups][EP_MAX_TOPK];
    __shared__ float s_coef_all[kGroups][EP_MAX_TOPK];
    __shared__ int s_n_all[kGroups];
    pdl_wait();
    if (kGroups == 1) {
        combine_item<kWeighted, kExpanded, 1, kB>(p, blockIdx.x, 0, threadIdx.x, s_rows_all[0], s_coef_all[0],
                                                  &s_n_all[0]);
    } else {
        const int group = static_cast<int>(threadIdx.x) / kThreads;
        const int gtid = static_cast<int>(threadIdx.x) % kThreads;
        const int64_t n_items = static_cast<int64_t>(p.T) * p.chunks;
        for (int64_t it = static_cast<int64_t>(blockIdx.x) * kGroups + group; it < n_items;
             it += static_cast<int64_t>(gridDim.x) * kGroups) {
            named_barrier(1 + group, kThreads);   // the previous item's list is consumed
            combine_item<kWeighted, kExpanded, kGroups, kB>(p, it, group, gtid, s_rows_all[group],
                                                            s_coef_all[group], &s_n_all[group]);
        }
    }
}

template <bool kWeighted, bool kExpanded>
cudaError_t launch_combine_t(const CombineParams& p, int64_t items, int num_sms, bool few, cudaStream_t stream) {
    if (num_sms > 0) {
        int64_t grid = (items + kSmGroups - 1) / kSmGroups;
        if (grid > num_sms) grid = num_sms;
        return launch_pdl(combine_kernel<kWeighted, kExpanded, kSmGroups, EP_COMBINE_SM_BATCH>,
                          dim3(static_cast<unsigned>(grid)), dim3(kThreads * kSmGroups), 0, stream, p);
    }
    if (few)
        return launch_pdl(combine_kernel<kWeighted, kExpanded, 1, EP_COMBINE_FEW_BATCH>,
                          dim3(static_cast<unsigned>(items)), dim3(kThreads), 0, stream, p);
    return launch_pdl(combine_kernel<kWeighted, kExpanded, 1, kBatch>, dim3(static_cast<unsigned>(items)),
                      dim3(kThreads), 0, stream, p);
}

}  // namespace

cudaError_t launch_combine(CombineParams p, bool weighted, cudaStream_t stream) {
    const DeviceInfo& di = device_info();
    const int n_vec = p.H / 8;
    const int num_sms = p.num_sms > 0 ? (p.num_sms < di.num_sms ? p.num_sms : di.num_sms) : 0;
    // Pieces of up to kCombineVecs (rank rows) or kCombineVecsExpanded
    // vectors per thread; more pieces when there are few tokens.  SM-limited: whole rows (each group's item then waits on one
    // routing load per row instead of one per quarter row: +40-55% at 16-64
    // SMs), unless there are fewer rows than groups.
    const int vecs = p.expanded_row ? kCombineVecsExpanded : kCombineVecs;
    int chunks = num_sms > 0 ? 1 : (n_vec + vecs * kThreads - 1) / (vecs * kThreads);
    const int64_t want_items = num_sms > 0 ? static_cast<int64_t>(num_sms) * kSmGroups : 4 * di.num_sms;
    const bool few = p.T > 0 && static_cast<int64_t>(p.T) * chunks < want_items;
    if (few) {
        // few tokens: latency-bound, so at most one vector per thread (each
        // CTA then waits for one batch of row loads per 4 rows, not two)
        int more = static_cast<int>((want_items + p.T - 1) / p.T);
        const int one_vec = (n_vec + kThreads - 1) / kThreads;
        if (more < one_vec) more = one_vec;
        const int max_chunks = (n_vec + 31) / 32;
        chunks = more < max_chunks ? more : max_chunks;
        if (chunks < 1) chunks = 1;
    }
    int chunk_vecs = (n_vec + chunks - 1) / chunks;
    chunks = (n_vec + chunk_vecs - 1) / chunk_vecs;
    p.chunks = chunks;
    p.chunk_vecs = chunk_vecs;
    const int64_t items = static_cast<int64_t>(p.T) * chunks;
    if (items < 1) return cudaSuccess;
    if (p.expanded_row) {
        if (weighted) return launch_combine_t<true, true>(p, items, num_sms, few, stream);
        return launch_combine_t<false, true>(p, items, num_sms, few, stream);
    }
    if (weighted) return launch_combine_t<true, false>(p, items, num_sms, few, stream);
    return launch_combine_t<false, false>(p, items, num_sms, few, stream);
}

}  // namespace epg
