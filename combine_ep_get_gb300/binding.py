"""ctypes binding of libep_get.so with the C ABI's entry-point names.

Argument marshalling only: tensors become device pointers, the current torch
CUDA stream becomes the cudaStream_t, and a non-zero host status raises.  All
computation happens in the library's CUDA kernels.  Importing this module
fails when the library has not been built (there is no CPU fallback).
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# EP_GET_LIBRARY names another build of the same library to load instead:
# the bounds-checked copy that the tests build (ep_bounds_checked() says which
# one is loaded).  Unset, the product library.
LIB_PATH = os.environ.get("EP_GET_LIBRARY") or os.path.join(_HERE, "libep_get.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("%s is not built; run `python -c \"import __graft_entry__ as g; "
                      "g.build()\"` or `python combine_ep_get_gb300/build.py`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_UNSUPPORTED = 2
EP_ERR_INVALID_INDEX = 4
EP_ERR_CAPACITY = 8
EP_ERR_TIMEOUT = 16
EP_ERR_CUDA = 32
EP_ERR_OUT_OF_BOUNDS = 64
EP_BF16 = 0
EP_FP8_E4M3 = 1

_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64


class ep_layout_t(ctypes.Structure):
    _fields_ = [("num_tokens_per_rank", _vp), ("num_tokens_per_node", _vp),
                ("num_tokens_per_expert", _vp), ("is_token_in_rank", _vp), ("rank_offset", _vp),
                ("expert_offset", _vp), ("dst_row", _vp), ("src_dst_count", _vp),
                ("token_offset", _vp), ("expanded_row", _vp), ("node_offset", _vp), ("node_row", _vp)]


_lib.ep_layout_workspace_bytes.restype = ctypes.c_size_t
_lib.ep_layout_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
_lib.ep_recv_capacity_bound.restype = _i64
_lib.ep_recv_capacity_bound.argtypes = [_i, _i, _i]
_lib.ep_get_layout.restype = ctypes.c_int32
_lib.ep_get_layout.argtypes = [_vp, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t), _vp,
                               ctypes.c_size_t, _vp, _vp]
_lib.ep_get_layout_static_scratch.restype = ctypes.c_int32
_lib.ep_get_layout_static_scratch.argtypes = [_vp, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t),
                                              _vp, _vp]
_lib.ep_dispatch.restype = ctypes.c_int32
_lib.ep_dispatch.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t), _i,
                             _i64, _vp, _vp, _i, _vp, _vp, _vp, _i, _vp, _vp]
_lib.ep_layout_and_dispatch.restype = ctypes.c_int32
_lib.ep_layout_and_dispatch.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t), _vp,
                                        ctypes.c_size_t, _i, _i64, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp]
_lib.ep_combine.restype = ctypes.c_int32
_lib.ep_combine.argtypes = [_vp, _i64, _vp, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t),
                            _vp, _i, _vp, _vp]
_lib.ep_expanded_capacity_bound.restype = _i64
_lib.ep_expanded_capacity_bound.argtypes = [_i, _i, _i, _i]
_lib.ep_dispatch_expanded.restype = ctypes.c_int32
_lib.ep_dispatch_expanded.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t), _i,
                                      _i64, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp]
_lib.ep_combine_expanded.restype = ctypes.c_int32
_lib.ep_combine_expanded.argtypes = [_vp, _i64, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t), _vp,
                                     _i, _vp, _vp]
_lib.ep_combine_topk_weights.restype = ctypes.c_int32
_lib.ep_combine_topk_weights.argtypes = [_vp, _i64, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t), _vp, _vp,
                                         _vp]
_lib.ep_accumulate_expert_stats.restype = ctypes.c_int32
_lib.ep_accumulate_expert_stats.argtypes = [ctypes.POINTER(ep_layout_t), _i, _vp, _vp]
_lib.ep_status_string.restype = ctypes.c_char_p
_lib.ep_status_string.argtypes = [ctypes.c_int32]
_lib.ep_abi_version.restype = _i
_lib.ep_abi_version.argtypes = []
_lib.ep_bounds_checked.restype = _i
_lib.ep_bounds_checked.argtypes = []
_lib.ep_dispatch_hierarchical.restype = ctypes.c_int32
_lib.ep_dispatch_hierarchical.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t), _i,
                                          _i64, _vp, _vp, _vp, _i64, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp]
_lib.ep_combine_hierarchical.restype = ctypes.c_int32
_lib.ep_combine_hierarchical.argtypes = [_vp, _i64, _vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ep_layout_t),
                                         _i64, _vp, _vp, _vp, _vp]
_lib.ep_theoretical_num_sms.restype = _i
_lib.ep_theoretical_num_sms.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_double, _i, _i]


def library():
    """The loaded ctypes library (for callers that marshal raw pointers)."""
    return _lib


def ep_bounds_checked() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(_lib.ep_bounds_checked())


def _ptr(t):
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(code, what):
    if code != EP_OK:
        raise RuntimeError("%s failed: %s" % (what, ep_status_string(code)))
    return code


def ep_status_string(status) -> str:
    return _lib.ep_status_string(int(status)).decode()


def ep_layout_workspace_bytes(num_tokens, num_topk, num_experts, num_ranks, ranks_per_node=0) -> int:
    return int(_lib.ep_layout_workspace_bytes(num_tokens, num_topk, num_experts, num_ranks,
                                              ranks_per_node))


def ep_recv_capacity_bound(num_tokens, num_topk, num_ranks) -> int:
    return int(_lib.ep_recv_capacity_bound(num_tokens, num_topk, num_ranks))


def ep_theoretical_num_sms(hidden, num_topk, num_experts, num_ranks, hbm_gbs, out_dtype=EP_BF16,
                           is_combine=False, sm_read_gbs=200.0, sm_write_gbs=50.0,
                           prefer_overlap_with_compute=True, device_sms=None) -> int:
    """SM count for the SM-limited mode; device_sms defaults to the current
    device's SM count.  Raises ValueError for arguments the library rejects."""
    if device_sms is None:
        device_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    n = int(_lib.ep_theoretical_num_sms(hidden, num_topk, num_experts, num_ranks, out_dtype, int(is_combine),
                                        float(hbm_gbs), float(sm_read_gbs), float(sm_write_gbs),
                                        int(prefer_overlap_with_compute), int(device_sms)))
    if n == 0:
        raise ValueError("ep_theoretical_num_sms: invalid arguments")
    return n


class Layout:
    """Device tensors of one routing layout plus their ep_layout_t view."""

    def __init__(self, T, E, R, ranks_per_node=0, with_src_dst=True, device="cuda", K=None, node_rows=False):
        i32 = dict(dtype=torch.int32, device=device)
        nodes = R // ranks_per_node if ranks_per_node > 0 else 0
        self.T, self.E, self.R, self.ranks_per_node = T, E, R, ranks_per_node
        self.num_tokens_per_rank = torch.empty(R, **i32)
        self.num_tokens_per_node = torch.empty(nodes, **i32) if nodes else None
        self.num_tokens_per_expert = torch.empty(E, **i32)
        self.is_token_in_rank = torch.empty((T, R), dtype=torch.uint8, device=device)
        self.rank_offset = torch.empty(R + 1, **i32)
        self.expert_offset = torch.empty(E + 1, **i32)
        self.dst_row = torch.empty((T, R), **i32)
        self.src_dst_count = torch.empty((R, R), **i32) if (with_src_dst and T % R == 0) else None
        self.token_offset = torch.empty(T + 1, **i32)
        # expanded (per-expert) rows are produced when K is given
        self.expanded_row = torch.empty((T, K), **i32) if K is not None else None
        # per-node scale-out rows (hierarchical path) when node_rows is set
        self.node_offset = torch.empty(nodes + 1, **i32) if (node_rows and nodes) else None
        self.node_row = torch.empty((T, nodes), **i32) if (node_rows and nodes) else None
        self.c = ep_layout_t(*[_ptr(getattr(self, f)) for f, _ in ep_layout_t._fields_])

    @property
    def num_recv(self) -> int:
        """N = rank_offset[R] (one device-to-host read)."""
        return int(self.rank_offset[-1].item())


def alloc_layout(T, E, R, ranks_per_node=0, with_src_dst=True, device="cuda", K=None, node_rows=False) -> Layout:
    """Device arrays of a layout; pass K to also get the expanded rows, and
    node_rows=True (with ranks_per_node > 0) for the hierarchical path's node rows."""
    return Layout(T, E, R, ranks_per_node, with_src_dst, device, K, node_rows)


def ep_expanded_capacity_bound(num_tokens, num_topk, num_experts, expert_alignment=1) -> int:
    return int(_lib.ep_expanded_capacity_bound(num_tokens, num_topk, num_experts, expert_alignment))


def ep_get_layout(topk_idx, num_experts, num_ranks, layout, workspace, d_status, ranks_per_node=0,
                  expert_alignment=1, stream=None):
    T, K = topk_idx.shape
    assert topk_idx.dtype == torch.int64 and topk_idx.is_contiguous()
    code = _lib.ep_get_layout(_ptr(topk_idx), T, K, num_experts, num_ranks, ranks_per_node,
                              expert_alignment, ctypes.byref(layout.c), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(d_status),
                              _stream(stream))
    return _check(code, "ep_get_layout")


def ep_get_layout_static_scratch(topk_idx, num_experts, num_ranks, layout, d_status, ranks_per_node=0,
                                 expert_alignment=1, stream=None):
    """ep_get_layout using the library's built-in scratch instead of a caller
    workspace, for callers that cannot allocate device memory (see the C
    header for the size limit and the ordering rule)."""
    T, K = topk_idx.shape
    assert topk_idx.dtype == torch.int64 and topk_idx.is_contiguous()
    code = _lib.ep_get_layout_static_scratch(_ptr(topk_idx), T, K, num_experts, num_ranks,
                                             ranks_per_node, expert_alignment, ctypes.byref(layout.c),
                                             _ptr(d_status), _stream(stream))
    return _check(code, "ep_get_layout_static_scratch")


def ep_dispatch(x, topk_idx, topk_weights, num_experts, num_ranks, layout, recv_x, recv_topk_idx,
                recv_topk_weights, recv_src_idx, d_status, recv_sf=None, out_dtype=EP_BF16,
                sf_col_major=False, num_sms=0, stream=None):
    T, H = x.shape
    K = topk_idx.shape[1]
    assert x.element_size() == 2 and x.is_contiguous() and recv_x.is_contiguous()
    capacity = recv_x.shape[0]
    code = _lib.ep_dispatch(_ptr(x), _ptr(topk_idx), _ptr(topk_weights), T, H, K, num_experts,
                            num_ranks, ctypes.byref(layout.c), out_dtype, capacity, _ptr(recv_x),
                            _ptr(recv_sf), 1 if sf_col_major else 0, _ptr(recv_topk_idx),
                            _ptr(recv_topk_weights), _ptr(recv_src_idx), num_sms, _ptr(d_status),
                            _stream(stream))
    return _check(code, "ep_dispatch")


def ep_dispatch_expanded(x, topk_idx, topk_weights, num_experts, num_ranks, layout, recv_x, recv_src_idx,
                         recv_weight, d_status, recv_sf=None, out_dtype=EP_BF16, sf_col_major=False,
                         num_sms=0, stream=None):
    T, H = x.shape
    K = topk_idx.shape[1]
    assert x.element_size() == 2 and x.is_contiguous() and recv_x.is_contiguous()
    code = _lib.ep_dispatch_expanded(_ptr(x), _ptr(topk_idx), _ptr(topk_weights), T, H, K, num_experts,
                                     num_ranks, ctypes.byref(layout.c), out_dtype, recv_x.shape[0],
                                     _ptr(recv_x), _ptr(recv_sf), 1 if sf_col_major else 0,
                                     _ptr(recv_src_idx), _ptr(recv_weight), num_sms, _ptr(d_status),
                                     _stream(stream))
    return _check(code, "ep_dispatch_expanded")


def ep_combine_expanded(y, topk_weights, num_topk, num_experts, num_ranks, layout, out, d_status,
                        num_sms=0, stream=None):
    T, H = out.shape
    assert y.element_size() == 2 and y.is_contiguous() and out.is_contiguous()
    code = _lib.ep_combine_expanded(_ptr(y), y.shape[0], _ptr(topk_weights), T, H, num_topk, num_experts,
                                    num_ranks, ctypes.byref(layout.c), _ptr(out), num_sms, _ptr(d_status),
                                    _stream(stream))
    return _check(code, "ep_combine_expanded")


def ep_combine_topk_weights(recv_topk_weights, num_experts, num_ranks, layout, combined, d_status,
                            stream=None):
    T, K = combined.shape
    assert recv_topk_weights.is_contiguous() and combined.is_contiguous()
    code = _lib.ep_combine_topk_weights(_ptr(recv_topk_weights), recv_topk_weights.shape[0], T, K,
                                        num_experts, num_ranks, ctypes.byref(layout.c), _ptr(combined),
                                        _ptr(d_status), _stream(stream))
    return _check(code, "ep_combine_topk_weights")


def ep_accumulate_expert_stats(layout, num_experts, stats, stream=None):
    assert stats.dtype == torch.int64 and stats.is_contiguous()
    code = _lib.ep_accumulate_expert_stats(ctypes.byref(layout.c), num_experts, _ptr(stats), _stream(stream))
    return _check(code, "ep_accumulate_expert_stats")


def ep_layout_and_dispatch(x, topk_idx, topk_weights, num_experts, num_ranks, layout, workspace, recv_x,
                           recv_topk_idx, recv_topk_weights, recv_src_idx, d_status, recv_sf=None,
                           out_dtype=EP_BF16, sf_col_major=False, ranks_per_node=0, expert_alignment=1,
                           stream=None):
    """ep_get_layout and ep_dispatch in one call (see the C header): one kernel
    for few tokens, else the layout kernel and the dispatch, whose first wave
    starts on the layout's rows-ready signal in `workspace`.  Size `workspace`
    with ep_layout_workspace_bytes and the receive arrays with
    ep_recv_capacity_bound; the workspace belongs to the call until the
    dispatch completes."""
    T, H = x.shape
    K = topk_idx.shape[1]
    assert x.element_size() == 2 and x.is_contiguous() and recv_x.is_contiguous()
    assert topk_idx.dtype == torch.int64 and topk_idx.is_contiguous()
    code = _lib.ep_layout_and_dispatch(_ptr(x), _ptr(topk_idx), _ptr(topk_weights), T, H, K, num_experts, num_ranks,
                                       ranks_per_node, expert_alignment, ctypes.byref(layout.c), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), out_dtype, recv_x.shape[0],
                                       _ptr(recv_x), _ptr(recv_sf), 1 if sf_col_major else 0, _ptr(recv_topk_idx),
                                       _ptr(recv_topk_weights), _ptr(recv_src_idx), _ptr(d_status), _stream(stream))
    return _check(code, "ep_layout_and_dispatch")


def ep_combine(y, topk_idx, topk_weights, num_experts, num_ranks, layout, out, d_status, num_sms=0,
               stream=None):
    T, H = out.shape
    K = topk_idx.shape[1]
    assert y.element_size() == 2 and y.is_contiguous() and out.is_contiguous()
    code = _lib.ep_combine(_ptr(y), y.shape[0], _ptr(topk_idx), _ptr(topk_weights), T, H, K,
                           num_experts, num_ranks, ctypes.byref(layout.c), _ptr(out), num_sms,
                           _ptr(d_status), _stream(stream))
    return _check(code, "ep_combine")


def ep_dispatch_hierarchical(x, topk_idx, topk_weights, num_experts, num_ranks, ranks_per_node, layout, node_x,
                             recv_x, d_status, node_sf=None, node_src_idx=None, recv_sf=None, recv_topk_idx=None,
                             recv_topk_weights=None, recv_src_idx=None, out_dtype=EP_BF16, sf_col_major=False,
                             stream=None):
    """Two-stage dispatch: node_x / node_sf / node_src_idx are the per-node
    scale-out buffers (node_capacity = node_x.shape[0]); recv_* as ep_dispatch."""
    T, H = x.shape
    K = topk_idx.shape[1]
    assert x.element_size() == 2 and x.is_contiguous() and recv_x.is_contiguous() and node_x.is_contiguous()
    code = _lib.ep_dispatch_hierarchical(_ptr(x), _ptr(topk_idx), _ptr(topk_weights), T, H, K, num_experts,
                                         num_ranks, ranks_per_node, ctypes.byref(layout.c), out_dtype,
                                         node_x.shape[0], _ptr(node_x), _ptr(node_sf), _ptr(node_src_idx),
                                         recv_x.shape[0], _ptr(recv_x), _ptr(recv_sf), int(sf_col_major),
                                         _ptr(recv_topk_idx), _ptr(recv_topk_weights), _ptr(recv_src_idx),
                                         _ptr(d_status), _stream(stream))
    return _check(code, "ep_dispatch_hierarchical")


def ep_combine_hierarchical(y, topk_idx, topk_weights, num_experts, num_ranks, ranks_per_node, layout, node_y,
                            out, d_status, stream=None):
    """Two-stage combine: node_y (bf16 [node_capacity, H]) receives the
    per-(token, node) partials; out the combined rows."""
    T, K = topk_idx.shape
    H = out.shape[1]
    assert y.element_size() == 2 and out.element_size() == 2 and node_y.element_size() == 2
    code = _lib.ep_combine_hierarchical(_ptr(y), y.shape[0], _ptr(topk_idx), _ptr(topk_weights), T, H, K,
                                        num_experts, num_ranks, ranks_per_node, ctypes.byref(layout.c),
                                        node_y.shape[0], _ptr(node_y), _ptr(out), _ptr(d_status), _stream(stream))
    return _check(code, "ep_combine_hierarchical")
