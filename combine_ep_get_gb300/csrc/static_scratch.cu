// ep_get_layout_static_scratch: the routing layout for callers that cannot
// allocate device memory.
//
// ep_get_layout needs a caller-provided device workspace.  Some callers have
// no way to provide one: a plugin that is handed only its input and output
// buffers by a host framework and owns no allocator, or a process whose device
// memory is fully reserved up front by a pooling allocator, where a further
// cudaMalloc fails or is not allowed once serving has started.  This entry
// point serves them: the workspace is a file-scope device array compiled into
// the library, so the call allocates nothing.  It forwards to ep_get_layout
// with that array as the workspace; results are identical.
#include <mutex>

#include "ep_internal.cuh"

namespace {

// The scratch array.  Every GPU that loads this library holds
// EP_LAYOUT_STATIC_SCRATCH_BYTES of it until the process exits.  In host code
// the name `g_layout_scratch` is only a host-side stand-in, never a device
// address: host code must use the address from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_layout_scratch[EP_LAYOUT_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device, resolved once
// per device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ep_status_t ep_get_layout_static_scratch(const int64_t* topk_idx, int num_tokens,
                                                    int num_topk, int num_experts, int num_ranks,
                                                    int ranks_per_node, int expert_alignment,
                                                    const ep_layout_t* out, int32_t* d_status,
                                                    void* cuda_stream) {
    if (num_tokens < 0 || num_experts < 1 || num_ranks < 1 || ranks_per_node < 0)
        return EP_ERR_INVALID_ARG;
    const size_t need =
        ep_layout_workspace_bytes(num_tokens, num_topk, num_experts, num_ranks, ranks_per_node);
    if (need > EP_LAYOUT_STATIC_SCRATCH_BYTES) return EP_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return EP_ERR_CUDA;
    return ep_get_layout(topk_idx, num_tokens, num_topk, num_experts, num_ranks, ranks_per_node,
                         expert_alignment, out, scratch, EP_LAYOUT_STATIC_SCRATCH_BYTES, d_status,
                         cuda_stream);
}
