"""The bounded-wait failure path of the bulk-copy dispatch ("DeepEP V2
ElasticBuffer architecture", the barrier fragment's timeout_while; "DeepEP
Symmetric Memory" section 9.1, num_gpu_timeout_secs), without faulting or
hanging the GPU.

A test-only copy of the library is built with a 1 ms wait limit and one
injected failure: CTA 0 of the bulk-copy dispatch (the SM-limited bf16 path)
announces its first row load on the slot's mbarrier and never issues it.
Nothing is in flight for that slot and every access stays in bounds; the wait
on it runs out, the kernel sets EP_ERR_TIMEOUT, drains its other loads and
stores (each wait again bounded) and returns.  The test checks the status
bit, that the kernel returned, and that the same stream then runs a normal
layout -> dispatch -> combine of the product library whose results match the
oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def _wait_test_library(B):
    from combine_ep_get_gb300 import build
    path = build.build_variant("waittest", ["-DEP_WAIT_TIMEOUT_NS=1000000ull", "-DEP_TEST_DROP_FIRST_LOAD"])
    lib = ctypes.CDLL(path)
    lib.ep_dispatch.restype = B.library().ep_dispatch.restype
    lib.ep_dispatch.argtypes = B.library().ep_dispatch.argtypes
    return lib


def test_dispatch_wait_runs_out_then_the_stream_works():
    from gpu_path import B, bf16_bits, run_combine, run_dispatch, run_layout, to_dev, x_tensor
    # T >= 2 * SMs: whole-row items split over the 4 CTAs by row number, so
    # CTA 0 owns a contiguous range of rows
    T, H, E, K, R = 320, 2048, 64, 6, 8
    d = make_inputs(T, H, E, K, R, seed=5)
    idx, w, x = to_dev(d["topk_idx"]), to_dev(d["topk_weights"]), x_tensor(d["x_bits"])
    lay, st = run_layout(idx, E, R)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    n = lay.num_recv
    rx = torch.zeros((n, H), dtype=torch.bfloat16, device="cuda")
    rs = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = _wait_test_library(B)
    stream = torch.cuda.current_stream()
    code = lib.ep_dispatch(x.data_ptr(), idx.data_ptr(), w.data_ptr(), T, H, K, E, R, ctypes.byref(lay.c),
                           B.EP_BF16, n, rx.data_ptr(), None, 0, None, None, rs.data_ptr(), 4,
                           status.data_ptr(), stream.cuda_stream)
    assert code == B.EP_OK
    stream.synchronize()                      # the kernel returned
    assert int(status.item()) & B.EP_ERR_TIMEOUT
    # CTA 0 gave up on its first row and stored none of its rows; the other
    # CTAs' rows are the oracle's
    L = oracle.layout(d["topk_idx"], E, R)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row)
    got = bf16_bits(rx).view(np.uint8).reshape(n, 2 * H)
    empty = ~got.any(axis=1)
    assert empty.any()
    np.testing.assert_array_equal(got[~empty], o["recv_x"][~empty])
    # the context is intact: a normal step on the same stream, product library
    lay2, st2 = run_layout(idx, E, R)
    res = run_dispatch(x, idx, w, E, R, lay2, n)
    out, st3 = run_combine(res["recv_x"], idx, None, E, R, lay2, T, H)
    torch.cuda.synchronize()
    assert int(st2.item()) == int(res["status"].item()) == int(st3.item()) == 0
    np.testing.assert_array_equal(lay2.dst_row.cpu().numpy(), L.dst_row)
    np.testing.assert_array_equal(bf16_bits(res["recv_x"][:n]).view(np.uint8).reshape(n, 2 * H), o["recv_x"])
    nt = lay2.is_token_in_rank.sum(dim=1, dtype=torch.int32).float()
    assert torch.equal(out.float(), (x.float() * nt[:, None]).to(torch.bfloat16).float())
