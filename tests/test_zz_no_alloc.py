"""ep_get_layout_static_scratch: the routing layout for callers that cannot
allocate device memory (a plugin handed only its input and output buffers, or
a process whose device memory is all reserved up front by a pooling
allocator).  It uses a device array built into the library instead of a
caller workspace.

Called here through the C ABI (ctypes) several times in a row on different
inputs -- a smaller call after a larger one too, which finds the most stale
scratch -- each result checked against the workspace entry point
ep_get_layout on the same input (integer outputs: exact).  This file is
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_ep_get_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

FIELDS = ("num_tokens_per_rank", "num_tokens_per_node", "num_tokens_per_expert", "is_token_in_rank",
          "rank_offset", "expert_offset", "dst_row", "src_dst_count", "token_offset")


def _static_layout(B, idx, E, R, rpn):
    T, K = idx.shape
    lay = B.alloc_layout(T, E, R, rpn)
    for f in FIELDS:
        t = getattr(lay, f)
        if t is not None:
            t.fill_(-5)                    # stale values must be overwritten
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = B.library().ep_get_layout_static_scratch
    code = fn(ctypes.c_void_p(idx.data_ptr()), T, K, E, R, rpn, 1, ctypes.byref(lay.c),
              ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == B.EP_OK, B.ep_status_string(code)
    return lay, status


def test_static_scratch_matches_workspace_entry_point_twice():
    from gpu_path import B, layout_host, run_layout, to_dev
    cases = [
        (4096, 8, 256, 8, 0, 1),           # DeepSeek-V3-shaped routing
        (32768, 8, 256, 64, 8, 2),         # large, node counts, src x dst counts
        (128, 8, 256, 32, 0, 3),           # smaller after larger: decode-shaped, single-CTA path
    ]
    for T, K, E, R, rpn, seed in cases:
        idx = to_dev(make_inputs(T, 8, E, K, R, seed=seed, mask_frac=0.03, with_x=False)["topk_idx"])
        ref_lay, ref_st = run_layout(idx, E, R, rpn)
        got_lay, got_st = _static_layout(B, idx, E, R, rpn)
        torch.cuda.synchronize()
        ref, got = layout_host(ref_lay), layout_host(got_lay)
        for f in FIELDS:
            if ref[f] is None:
                assert got[f] is None
            else:
                np.testing.assert_array_equal(got[f], ref[f], err_msg=f)
        assert int(got_st.item()) == int(ref_st.item()) == 0


def test_static_scratch_rejects_sizes_beyond_its_array():
    from gpu_path import B
    T, K, E, R = 65536, 8, 2048, 1024
    assert B.ep_layout_workspace_bytes(T, K, E, R, 0) > (4 << 20)
    # valid-looking 16-byte-aligned stand-in addresses: every argument check
    # passes, the size check rejects the call before anything is launched
    vp = ctypes.c_void_p
    lay = B.ep_layout_t(16, None, 32, 48, 64, 80, 96, None, None)
    fn = B.library().ep_get_layout_static_scratch
    code = fn(vp(16), T, K, E, R, 0, 1, ctypes.byref(lay), vp(16), None)
    assert code == B.EP_ERR_UNSUPPORTED


def test_static_scratch_argument_errors_match_the_workspace_entry_point():
    """A bad argument gives the code ep_get_layout gives, even for sizes the
    built-in scratch could not hold (checked on the host, nothing launched)."""
    from gpu_path import B
    lay = B.ep_layout_t()
    st = ctypes.c_void_p(16)             # a stand-in device address; never dereferenced here
    fn = B.library().ep_get_layout_static_scratch
    for args in [(None, 10, 8, 256, 7, 0, 1),            # R does not divide E
                 (None, 65536, 8, 2048, 1024, 3, 1),     # too large, and rpn does not divide R
                 (None, 10, 33, 256, 8, 0, 1)]:          # top-33
        want = B.library().ep_get_layout(args[0], *args[1:], ctypes.byref(lay), None, 0, st, None)
        got = fn(args[0], *args[1:], ctypes.byref(lay), st, None)
        assert got == want != B.EP_OK
