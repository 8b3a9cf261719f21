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
#include "ep_internal.cuh"

namespace {

// The scratch array.  Every GPU that loads this library holds
// EP_LAYOUT_STATIC_SCRATCH_BYTES of it until the process exits.  In host code
// the name `g_layout_scratch` is only a host-side stand-in, never a device
// address: host code must use the address from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_layout_scratch[EP_LAYOUT_STATIC_SCRATCH_BYTES];

// Device address of g_layout_scratch on the current device, looked up on
// every call (with that device current; cheap, allocates nothing), so that it
// stays right if the device was reset and the module loaded again.
cudaError_t scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_layout_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" ep_status_t ep_get_layout_static_scratch(const int64_t* topk_idx, int num_tokens,
                                                    int num_topk, int num_experts, int num_ranks,
                                                    int ranks_per_node, int expert_alignment,
                                                    const ep_layout_t* out, int32_t* d_status,
                                                    void* cuda_stream) {
    // every argument check of ep_get_layout first, so a bad argument gives the
    // same code as there; then the size of the built-in scratch
    EP_DEBUG("ep_get_layout_static_scratch: T=%d K=%d E=%d R=%d", num_tokens, num_topk, num_experts, num_ranks);
    epg::LayoutParams unused{};
    const ep_status_t s = epg::layout_params(topk_idx, num_tokens, num_topk, num_experts, num_ranks,
                                             ranks_per_node, expert_alignment, out, nullptr, 0, d_status,
                                             false, unused);
    if (s != EP_OK) return s;
    const size_t need =
        ep_layout_workspace_bytes(num_tokens, num_topk, num_experts, num_ranks, ranks_per_node);
    if (need > EP_LAYOUT_STATIC_SCRATCH_BYTES) {
        EP_DEBUG("ep_get_layout_static_scratch: needs %zu bytes of scratch, has %zu: unsupported", need,
                 static_cast<size_t>(EP_LAYOUT_STATIC_SCRATCH_BYTES));
        return EP_ERR_UNSUPPORTED;
    }
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) {
        EP_DEBUG("ep_get_layout_static_scratch: cudaGetSymbolAddress failed");
        return EP_ERR_CUDA;
    }
    return ep_get_layout(topk_idx, num_tokens, num_topk, num_experts, num_ranks, ranks_per_node,
                         expert_alignment, out, scratch, EP_LAYOUT_STATIC_SCRATCH_BYTES, d_status,
                         cuda_stream);
}
