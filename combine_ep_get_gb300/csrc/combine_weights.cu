// Two small companions of combine:
//  - combined top-k weights ("DeepEP Symmetric Memory" section 9.2: combine
//    also returns combined_topk_weights): for token t and slot k, the fp32 sum
//    over the ranks holding t (ascending) of the received row's weight in slot
//    k.  One warp per token: lane r finds rank r's row, members are broadcast
//    by shuffles, lane k accumulates slot k.
//  - cumulative per-expert receive statistics (section 6.1:
//    cumulative_local_expert_recv_stats): stats[e] += num_tokens_per_expert[e].
#include "ep_internal.cuh"

namespace epg {
namespace {

constexpr int kWeightThreads = 256;

__global__ void __launch_bounds__(kWeightThreads) combine_topk_weights_kernel(const CombineWeightsParams p) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (kWeightThreads / 32) + (threadIdx.x >> 5);
    if (t >= p.T) return;
    float acc = 0.0f;
    bool cap_bad = false;
    for (int rb = 0; rb < p.R; rb += 32) {
        const int r = rb + lane;
        const int d = (r < p.R && EP_IN(t * p.R + r, static_cast<int64_t>(p.T) * p.R)) ? p.dst_row[t * p.R + r] : -1;
        (void)EP_ROW_OK(d);
        const bool ok = d >= 0 && d < p.num_rows;
        if (d >= p.num_rows) cap_bad = true;
        unsigned m = __ballot_sync(0xffffffffu, ok);
        while (m) {
            const int sl = __ffs(m) - 1;
            m &= m - 1u;
            const int64_t dd = __shfl_sync(0xffffffffu, d, sl);
            if (lane < p.K && EP_IN(dd * p.K + lane, p.num_rows * p.K)) acc += p.recv_topk_weights[dd * p.K + lane];
        }
    }
    if (lane < p.K && EP_IN(t * p.K + lane, static_cast<int64_t>(p.T) * p.K)) p.combined[t * p.K + lane] = acc;
    if (__any_sync(0xffffffffu, cap_bad) && lane == 0) atomicOr(p.status, EP_ERR_CAPACITY);
}

__global__ void accumulate_expert_stats_kernel(const int32_t* counts, int E, int64_t* stats) {
    pdl_wait();
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x)
        stats[e] += counts[e];
}

}  // namespace

cudaError_t launch_combine_topk_weights(const CombineWeightsParams& p, cudaStream_t stream) {
    const int64_t blocks = (static_cast<int64_t>(p.T) + kWeightThreads / 32 - 1) / (kWeightThreads / 32);
    if (blocks < 1) return cudaSuccess;
    return launch_pdl(combine_topk_weights_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kWeightThreads), 0,
                      stream, p);
}

cudaError_t launch_accumulate_expert_stats(const int32_t* counts, int E, int64_t* stats, cudaStream_t stream) {
    const int blocks = (E + 255) / 256;
    return launch_pdl(accumulate_expert_stats_kernel, dim3(blocks), dim3(256), 0, stream, counts, E, stats);
}

}  // namespace epg
