// Scale-up halves of the hierarchical (two-stage) path ("DeepEP V2
// ElasticBuffer architecture": hybrid_dispatch / hybrid_combine, used when
// there is more than one scale-out domain; node = rank / ranks_per_node as in
// "V1 Buffer initialisation" section 3.2).
//
// Dispatch stage 1 (scale-out) sends each token once to every node holding
// one of its experts: the ordinary dispatch kernels run with node_row as the
// destination table.  Stage 2 (here, forward_scaleup_kernel) copies each node
// row to the ranks of that node that need the token and writes the same
// per-row metadata as the single-stage dispatch, so the receive buffers come
// out identical.
//
// Combine stage 1 (here, reduce_scaleup_kernel) sums, per (token, node), the
// rows of the node's ranks (fp32, weighted or not) into one bf16 node row;
// stage 2 (scale-out) is the ordinary unweighted combine over node_row.
//
// Both kernels take one CTA per (token, piece); the forwarder walks the
// token's nodes in order, the reduce compacts all the token's source rows at
// once (ascending rank, hence grouped by node) and streams them in batches
// across node boundaries.  All stores are 16-byte vectors.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace epg {
namespace {

constexpr int kFwdThreads = 256;
constexpr int kFwdUnroll = 4;
constexpr int kRedThreads = 128;
constexpr int kRedBatch = 4;

// One of the receive-metadata arrays of token t's rows on ranks [r0, r1)
// (part 0: recv_topk_idx, 1: recv_topk_weights, 2: recv_src_idx), one warp
// (lane k < K).  The rows of up to 32 ranks are loaded at once, one per lane.
__device__ __forceinline__ void forward_metadata(const HierParams& p, int t, int r0, int r1, int lane, int part) {
    const int K = p.K;
    int64_t e_l = -1;
    float w_l = 0.0f;
    if (part < 2 && lane < K && EP_IN(static_cast<int64_t>(t) * K + lane, static_cast<int64_t>(p.T) * K)) {
        e_l = p.topk_idx[static_cast<int64_t>(t) * K + lane];
        if (part == 1 && p.recv_topk_weights) w_l = p.topk_weights[static_cast<int64_t>(t) * K + lane];
    }
    // the rank of this lane's expert and its index there, once (not per destination)
    const int e_rank = (e_l >= 0 && e_l < p.E) ? static_cast<int>(e_l) / p.experts_per_rank : -1;
    const int32_t e_local = static_cast<int32_t>(e_l) - e_rank * p.experts_per_rank;
    for (int rb = r0; rb < r1; rb += 32) {
        const int64_t dr = static_cast<int64_t>(t) * p.R + rb + lane;
        const int d = (rb + lane < r1 && EP_IN(dr, static_cast<int64_t>(p.T) * p.R)) ? p.dst_row[dr] : -1;
        (void)EP_ROW_OK(d);
        unsigned m = __ballot_sync(0xffffffffu, d >= 0 && d < p.capacity);
        while (m) {
            const int sl = __ffs(m) - 1;
            m &= m - 1;
            const int64_t dd = __shfl_sync(0xffffffffu, d, sl);
            const int r = rb + sl;
            if (part < 2) {
                if (lane < K && EP_IN(dd * K + lane, p.capacity * K)) {
                    const bool on = e_rank == r;
                    if (part == 0) {
                        if (p.recv_topk_idx) p.recv_topk_idx[dd * K + lane] = on ? e_local : -1;
                    } else if (p.recv_topk_weights) {
                        p.recv_topk_weights[dd * K + lane] = on ? w_l : 0.0f;
                    }
                }
            } else if (lane == 0 && p.recv_src_idx) {
                p.recv_src_idx[dd] = t;
            }
        }
    }
}

template <bool kFp8>
__global__ void __launch_bounds__(kFwdThreads, 6) forward_scaleup_kernel(const HierParams p) {
    const int gtid = threadIdx.x;
    const int warp = gtid >> 5;
    const int lane = gtid & 31;
    pdl_wait();   // node rows come from the previous kernel
    const int t = static_cast<int>(blockIdx.x / p.chunks);
    const int c = static_cast<int>(blockIdx.x - static_cast<unsigned>(t) * p.chunks);
    const uint32_t row_bytes = kFp8 ? static_cast<uint32_t>(p.H) : static_cast<uint32_t>(p.H) * 2u;
    const uint32_t off = static_cast<uint32_t>(c) * p.chunk_bytes;
    const int nvec = static_cast<int>(min(p.chunk_bytes, row_bytes - off) / 16);
    const int nb = p.H / 128;
    const int rpn = p.ranks_per_node;
    bool cap_bad = false;
    const int64_t row_in = static_cast<int64_t>(p.node_capacity) * row_bytes;
    const int64_t row_out = p.capacity * row_bytes;
    const uint64_t store_pol = l2_policy_evict_first();   // the rank rows stream out past L2
    // the token's node rows of the first 32 nodes, one per lane, in one load
    const int64_t nr0 = static_cast<int64_t>(t) * p.num_nodes, n_nr = static_cast<int64_t>(p.T) * p.num_nodes;
    const int j_lane = (lane < p.num_nodes && EP_IN(nr0 + lane, n_nr)) ? p.node_row[nr0 + lane] : -1;
    for (int n = 0; n < p.num_nodes; ++n) {
        const int j = n < 32 ? __shfl_sync(0xffffffffu, j_lane, n)
                             : (EP_IN(nr0 + n, n_nr) ? p.node_row[nr0 + n] : -1);   // uniform over the CTA
        (void)EP_ROW_OK(j);
        if (j < 0) continue;
        if (j >= p.node_capacity) {
            cap_bad = true;
            continue;
        }
        const int r0 = n * rpn;
        // receive metadata: one array per warp (1, 2, 3); FP8 scales: warp 4
        if (c == 0 && warp >= 1 && warp <= 3) forward_metadata(p, t, r0, r0 + rpn, lane, warp - 1);
        if (kFp8 && c == 0 && warp == 4 && p.recv_sf) {
            const int64_t sf_n = p.sf_col_major ? static_cast<int64_t>(nb) * p.sf_stride : p.capacity * nb;
            for (int rb = r0; rb < r0 + rpn; rb += 32) {
                const int64_t dr = static_cast<int64_t>(t) * p.R + rb + lane;
                const int d_l = (rb + lane < r0 + rpn && EP_IN(dr, static_cast<int64_t>(p.T) * p.R)) ? p.dst_row[dr] : -1;
                unsigned m = __ballot_sync(0xffffffffu, d_l >= 0 && d_l < p.capacity);
                while (m) {
                    const int sl = __ffs(m) - 1;
                    m &= m - 1;
                    const int d = __shfl_sync(0xffffffffu, d_l, sl);
                    for (int b = lane; b < nb; b += 32) {
                        if (!EP_IN(static_cast<int64_t>(j) * nb + b, static_cast<int64_t>(p.node_capacity) * nb)) continue;
                        const float s = p.node_sf[static_cast<int64_t>(j) * nb + b];
                        const int64_t si = p.sf_col_major ? static_cast<int64_t>(b) * p.sf_stride + d
                                                          : static_cast<int64_t>(d) * nb + b;
                        if (EP_IN(si, sf_n)) p.recv_sf[si] = s;
                    }
                }
            }
        }
        const int64_t src_off = static_cast<int64_t>(j) * row_bytes + off;
        const uint8_t* src = p.node_x + src_off;
        const int64_t drow0 = static_cast<int64_t>(t) * p.R + r0;
        const int32_t* drow = p.dst_row + drow0;
        for (int base = 0; base < nvec; base += kFwdUnroll * kFwdThreads) {
            uint4 u[kFwdUnroll];
#pragma unroll
            for (int k = 0; k < kFwdUnroll; ++k) {
                const int v = base + gtid + k * kFwdThreads;
                if (v < nvec && EP_IN_BYTES(src_off + static_cast<int64_t>(v) * 16, 16, row_in))
                    u[k] = ld_stream_v4(src + static_cast<size_t>(v) * 16);
            }
            for (int rb = 0; rb < rpn; rb += 32) {
                const int d = (rb + lane < rpn && EP_IN(drow0 + rb + lane, static_cast<int64_t>(p.T) * p.R))
                                  ? drow[rb + lane] : -1;
                (void)EP_ROW_OK(d);
                if (d >= p.capacity && c == 0 && base == 0) cap_bad = true;
                unsigned m = __ballot_sync(0xffffffffu, d >= 0 && d < p.capacity);
                while (m) {
                    const int sl = __ffs(m) - 1;
                    m &= m - 1;
                    const int64_t dst_off = static_cast<int64_t>(__shfl_sync(0xffffffffu, d, sl)) * row_bytes + off;
                    uint8_t* dst = p.recv_x + dst_off;
#pragma unroll
                    for (int k = 0; k < kFwdUnroll; ++k) {
                        const int v = base + gtid + k * kFwdThreads;
                        if (v < nvec && EP_IN_BYTES(dst_off + static_cast<int64_t>(v) * 16, 16, row_out))
                            st_v4_hint(dst + static_cast<size_t>(v) * 16, u[k], store_pol);
                    }
                }
            }
        }
    }
    // every warp sees the same rows; warp 0 of the first piece reports
    if (warp == 0 && c == 0 && __any_sync(0xffffffffu, cap_bad) && lane == 0) atomicOr(p.status, EP_ERR_CAPACITY);
}

template <bool kWeighted>
__global__ void __launch_bounds__(kRedThreads, 12) reduce_scaleup_kernel(const HierParams p) {
    __shared__ int s_rows[EP_MAX_TOPK];
    __shared__ float s_coef[EP_MAX_TOPK];
    __shared__ int s_dst[EP_MAX_TOPK];   // node row (partial) each source row adds into
    __shared__ int s_n;
    const int gtid = threadIdx.x;
    pdl_wait();
    const int t = static_cast<int>(blockIdx.x / p.chunks);
    const int c = static_cast<int>(blockIdx.x - static_cast<unsigned>(t) * p.chunks);
    const int rpn = p.ranks_per_node;
    // Warp 0: the token's source rows over all ranks in ascending order, which
    // groups them by node; each entry carries its node's row in node_y.
    if (gtid < 32) {
        const int lane = gtid;
        int64_t e_l = -1;
        float w_l = 0.0f;
        if (kWeighted && lane < p.K && EP_IN(static_cast<int64_t>(t) * p.K + lane, static_cast<int64_t>(p.T) * p.K)) {
            e_l = p.topk_idx[static_cast<int64_t>(t) * p.K + lane];
            w_l = p.topk_weights[static_cast<int64_t>(t) * p.K + lane];
        }
        const int32_t* nrow = p.node_row + static_cast<int64_t>(t) * p.num_nodes;
        const int j_lane = (lane < p.num_nodes && EP_IN(static_cast<int64_t>(t) * p.num_nodes + lane,
                                                        static_cast<int64_t>(p.T) * p.num_nodes))
                               ? nrow[lane]
                               : -1;   // nodes 0..31, with the rank rows
        const int32_t* srow = p.dst_row + static_cast<int64_t>(t) * p.R;
        int n = 0;
        bool cap_bad = false;
        for (int rb = 0; rb < p.R; rb += 32) {
            const int r = rb + lane;
            const int d = (r < p.R && EP_IN(static_cast<int64_t>(t) * p.R + r, static_cast<int64_t>(p.T) * p.R)) ? srow[r] : -1;
            (void)EP_ROW_OK(d);
            const int nd = r / rpn;
            int j = -1;
            if (nd < 32) {
                j = __shfl_sync(0xffffffffu, j_lane, nd & 31);
            } else if (d >= 0 && EP_IN(static_cast<int64_t>(t) * p.num_nodes + nd, static_cast<int64_t>(p.T) * p.num_nodes)) {
                j = nrow[nd];
            }
            // a row beyond num_y_rows stays in the list as a null entry (never
            // loaded), so its node's partial is still written from the others
            bool ok = d >= 0;
            if (d >= p.num_y_rows) cap_bad = true;
            if (ok && (j < 0 || j >= p.node_capacity)) {   // the node's partial row does not exist
                if (j >= p.node_capacity) cap_bad = true;
                ok = false;
            }
            float coef = 1.0f;
            if (kWeighted) {
                coef = 0.0f;
                for (int k = 0; k < p.K; ++k) {
                    const int64_t e = __shfl_sync(0xffffffffu, e_l, k);
                    const float w = __shfl_sync(0xffffffffu, w_l, k);
                    if (e >= 0 && e < p.E && static_cast<int>(e) / p.experts_per_rank == r) coef += w;
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, ok);
            const int pos = n + __popc(m & ((1u << lane) - 1u));
            if (ok && pos < EP_MAX_TOPK) {
                s_rows[pos] = d < p.num_y_rows ? d : -1;
                s_coef[pos] = coef;
                s_dst[pos] = j;
            }
            n += __popc(m);
        }
        if (n > EP_MAX_TOPK) {
            if (lane == 0) atomicOr(p.status, EP_ERR_INVALID_INDEX);
            n = EP_MAX_TOPK;
        }
        if (lane == 0) s_n = n;
        if (__any_sync(0xffffffffu, cap_bad) && lane == 0 && c == 0) atomicOr(p.status, EP_ERR_CAPACITY);
    }
    __syncthreads();

    const int n = s_n;
    const int n_vec = p.H / 8;
    const int v_begin = c * p.chunk_vecs;
    const int v_end = min(n_vec, v_begin + p.chunk_vecs);
    const int64_t row_bytes = static_cast<int64_t>(p.H) * 2;
    for (int v = v_begin + gtid; v < v_end; v += kRedThreads) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        const int64_t voff = static_cast<int64_t>(v) * 16;
        // rows of all the token's nodes in batches; a node's partial is stored
        // after its last row, then the sum restarts
        for (int m0 = 0; m0 < n; m0 += kRedBatch) {
            uint4 buf[kRedBatch];
#pragma unroll
            for (int i = 0; i < kRedBatch; ++i) {
                const int d = m0 + i < n ? s_rows[m0 + i] : -1;
                buf[i] = (d >= 0 && EP_IN_BYTES(static_cast<int64_t>(d) * row_bytes + voff, 16, p.num_y_rows * row_bytes))
                             ? ld_stream_v4(p.y + static_cast<int64_t>(d) * row_bytes + voff)
                             : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < kRedBatch; ++i) {
                const int m = m0 + i;
                if (m < n) {
                    const uint32_t w[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
                    const float cf = kWeighted ? s_coef[m] : 1.0f;
                    const bool live = s_rows[m] >= 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (!live) {
                        } else if (kWeighted) {
                            acc[2 * q] = fmaf(cf, __uint_as_float(w[q] << 16), acc[2 * q]);
                            acc[2 * q + 1] = fmaf(cf, __uint_as_float(w[q] & 0xffff0000u), acc[2 * q + 1]);
                        } else {
                            acc[2 * q] += __uint_as_float(w[q] << 16);
                            acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
                        }
                    }
                    const int j = s_dst[m];
                    if (m == n - 1 || s_dst[m + 1] != j) {
                        uint4 o;
                        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
                            ow[q] = *reinterpret_cast<const uint32_t*>(&h);
                            acc[2 * q] = 0.0f;
                            acc[2 * q + 1] = 0.0f;
                        }
                        if (EP_IN_BYTES(static_cast<int64_t>(j) * row_bytes + voff, 16, p.node_capacity * row_bytes))
                            st_v4(p.node_y + static_cast<int64_t>(j) * row_bytes + voff, o);
                    }
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_forward_scaleup(HierParams p, bool fp8, cudaStream_t stream) {
    const DeviceInfo& di = device_info();
    const uint32_t row_bytes = fp8 ? static_cast<uint32_t>(p.H) : static_cast<uint32_t>(p.H) * 2u;
    // pieces of at most 16 KB; more pieces when there are few tokens
    int chunks = static_cast<int>((row_bytes + 16383u) / 16384u);
    const int want_items = 4 * di.num_sms;
    if (p.T > 0 && static_cast<int64_t>(p.T) * chunks < want_items) {
        const int more = (want_items + p.T - 1) / p.T;
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
    const dim3 grid(static_cast<unsigned>(items)), block(kFwdThreads);
    if (fp8) return launch_pdl(forward_scaleup_kernel<true>, grid, block, 0, stream, p);
    return launch_pdl(forward_scaleup_kernel<false>, grid, block, 0, stream, p);
}

cudaError_t launch_reduce_scaleup(HierParams p, bool weighted, cudaStream_t stream) {
    const DeviceInfo& di = device_info();
    const int n_vec = p.H / 8;
    int chunks = (n_vec + 2 * kRedThreads - 1) / (2 * kRedThreads);
    const int want_items = 4 * di.num_sms;
    if (p.T > 0 && static_cast<int64_t>(p.T) * chunks < want_items) {
        const int more = (want_items + p.T - 1) / p.T;
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
    const dim3 grid(static_cast<unsigned>(items)), block(kRedThreads);
    if (weighted) return launch_pdl(reduce_scaleup_kernel<true>, grid, block, 0, stream, p);
    return launch_pdl(reduce_scaleup_kernel<false>, grid, block, 0, stream, p);
}

}  // namespace epg
