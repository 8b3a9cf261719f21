"""The bounds-checked build of the library: every kernel compiled with
EP_GET_CHECKED=1, ep_bounds_checked() == 1.

In that build each global load and store is tested against the extent its
call's arguments declare (T x R for dst_row, capacity x row bytes for the
receive buffer, and so on); an access that fails is skipped and sets
EP_ERR_OUT_OF_BOUNDS in the status word.  Nothing traps.  Two kinds of test:

* the whole GPU suite again, in a child process that loads the checked copy
  (EP_GET_LIBRARY): every parity test there asserts status 0 and the oracle's
  results, so on valid input no check fires;
* malformed row tables (an entry below -1 in dst_row, expanded_row or
  node_row) given to the rank-row, expanded and two-stage dispatch and to the
  rank-row and expanded combine, run under both builds: the checked build
  reports EP_ERR_OUT_OF_BOUNDS, the product build reads the entry as absent
  (as -1) with status 0; every other row is the oracle's under both.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import make_inputs, make_rows
from tolerance import check_close, combine_bounds, expanded_sources, rank_combine_bounds

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpu_suite_under_the_bounds_checked_build():
    from gpu_path import B
    if B.ep_bounds_checked():
        pytest.skip("this process already runs the checked build")
    from combine_ep_get_gb300 import build
    path = build.build_variant("checked", ["-DEP_GET_CHECKED=1"], recompile="all")
    env = dict(os.environ, EP_GET_LIBRARY=path)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-6000:] + r.stderr[-3000:]
    assert " passed" in r.stdout and " failed" not in r.stdout


def test_the_loaded_build_is_the_one_asked_for():
    from gpu_path import B
    assert B.ep_bounds_checked() == bool(os.environ.get("EP_GET_LIBRARY"))


def _expect(B, status):
    want = B.EP_ERR_OUT_OF_BOUNDS if B.ep_bounds_checked() else 0
    assert int(status.item()) == want, B.ep_status_string(int(status.item()))


def _plant(dst_row, value, seed):
    """Replace a few present entries of a row table by `value`; returns the
    table as the product reads it (those entries -1) and the dropped rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    present = np.argwhere(dst_row >= 0)
    pick = present[rng.choice(len(present), size=min(5, len(present)), replace=False)]
    bad, read_as = dst_row.copy(), dst_row.copy()
    dropped = []
    for i, j in pick:
        dropped.append(int(dst_row[i, j]))
        bad[i, j] = value
        read_as[i, j] = -1
    return bad, read_as, np.array(dropped)


@pytest.mark.parametrize("mode", ["bf16", "fp8", "bulk"])
def test_dispatch_with_rows_below_minus_one(mode):
    from gpu_path import B, bf16_bits, run_layout, to_dev, x_tensor
    T, H, E, K, R = 320, 1024, 64, 6, 8
    d = make_inputs(T, H, E, K, R, seed=21)
    idx, w, x = to_dev(d["topk_idx"]), to_dev(d["topk_weights"]), x_tensor(d["x_bits"])
    lay, st = run_layout(idx, E, R)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    n = lay.num_recv
    L = oracle.layout(d["topk_idx"], E, R)
    bad, read_as, dropped = _plant(L.dst_row, -5, seed=3)
    lay.dst_row.copy_(torch.from_numpy(bad))
    fp8 = mode == "fp8"
    rx = (torch.full((n, H), 0x55, dtype=torch.uint8, device="cuda") if fp8
          else torch.full((n, H), -3.0, dtype=torch.bfloat16, device="cuda"))
    rsf = torch.full((n * (H // 128),), -1.0, dtype=torch.float32, device="cuda") if fp8 else None
    rs = torch.full((n,), -9, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_dispatch(x, idx, w, E, R, lay, rx, None, None, rs, status, recv_sf=rsf,
                  out_dtype=B.EP_FP8_E4M3 if fp8 else B.EP_BF16, num_sms=4 if mode == "bulk" else 0)
    torch.cuda.synchronize()
    _expect(B, status)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, read_as, capacity=n, fp8=fp8)
    keep = np.ones(n, bool)
    keep[dropped] = False
    got = rx.cpu().numpy().view(np.uint8).reshape(n, -1) if fp8 else bf16_bits(rx).view(np.uint8).reshape(n, 2 * H)
    np.testing.assert_array_equal(got[keep], o["recv_x"][keep])
    np.testing.assert_array_equal(rs.cpu().numpy()[keep], o["recv_src_idx"][keep])
    assert (rs.cpu().numpy()[dropped] == -9).all()     # the dropped rows were never written
    if fp8:
        np.testing.assert_array_equal(rsf.cpu().numpy().reshape(n, -1)[keep], o["recv_sf"][keep])


@pytest.mark.parametrize("weighted", [False, True])
def test_combine_with_rows_below_minus_one(weighted):
    from gpu_path import B, bf16_bits, run_layout, to_dev
    T, H, E, K, R = 300, 2048, 64, 6, 8
    d = make_inputs(T, 8, E, K, R, seed=23, with_x=False)
    idx, w = to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    lay, st = run_layout(idx, E, R)
    torch.cuda.synchronize()
    n = lay.num_recv
    L = oracle.layout(d["topk_idx"], E, R)
    bad, read_as, _ = _plant(L.dst_row, -2, seed=4)
    lay.dst_row.copy_(torch.from_numpy(bad))
    y_bits = make_rows(n, H, seed=5)
    y = to_dev(y_bits.view(np.int16), torch.bfloat16)
    out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_combine(y, idx, w if weighted else None, E, R, lay, out, status)
    torch.cuda.synchronize()
    _expect(B, status)
    ref, _ = oracle.combine(y_bits, d["topk_idx"], d["topk_weights"], E, R, read_as, weighted=weighted)
    loose, tight = rank_combine_bounds(y_bits, d["topk_idx"], d["topk_weights"], E, R, read_as, weighted, ref)
    check_close(bf16_bits(out), ref, loose, tight)


def test_expanded_combine_with_rows_below_minus_one():
    from gpu_path import B, bf16_bits, to_dev
    T, H, E, K, R = 256, 1024, 64, 6, 8
    d = make_inputs(T, 8, E, K, R, seed=27, with_x=False)
    idx, w = to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    lay = B.alloc_layout(T, E, R, 0, K=K)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, 0), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, st, 0, 1)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = lay.expanded_row.cpu().numpy()
    n = int(rows.max()) + 1
    bad, read_as, _ = _plant(rows, -9, seed=6)
    lay.expanded_row.copy_(torch.from_numpy(bad))
    y_bits = make_rows(n, H, seed=7)
    y = to_dev(y_bits.view(np.int16), torch.bfloat16)
    out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_combine_expanded(y, w, K, E, R, lay, out, status)
    torch.cuda.synchronize()
    _expect(B, status)
    ref, _ = oracle.combine_expanded(y_bits, d["topk_weights"], read_as, weighted=True)
    src_rows, c, a, m = expanded_sources(read_as, d["topk_weights"], True)
    loose, tight = combine_bounds(y_bits, src_rows, c, a, ref, m)
    check_close(bf16_bits(out), ref, loose, tight)


def test_expanded_dispatch_with_rows_below_minus_one():
    from gpu_path import B, bf16_bits, to_dev, x_tensor
    T, H, E, K, R = 200, 1024, 64, 6, 8
    d = make_inputs(T, H, E, K, R, seed=29)
    idx, w = to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    lay = B.alloc_layout(T, E, R, 0, K=K)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, 0), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, st, 0, 1)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    cap = int(lay.expert_offset[-1].item())
    bad, read_as, dropped = _plant(lay.expanded_row.cpu().numpy(), -4, seed=8)
    lay.expanded_row.copy_(torch.from_numpy(bad))
    rx = torch.full((cap, H), -3.0, dtype=torch.bfloat16, device="cuda")
    rs = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    rw = torch.full((cap,), -9.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_dispatch_expanded(x_tensor(d["x_bits"]), idx, w, E, R, lay, rx, rs, rw, status)
    torch.cuda.synchronize()
    _expect(B, status)
    o = oracle.dispatch_expanded(d["x_bits"], d["topk_weights"], read_as, cap)
    valid = np.unique(read_as[read_as >= 0])
    np.testing.assert_array_equal(bf16_bits(rx).view(np.uint8).reshape(cap, 2 * H)[valid], o["recv_x"][valid])
    np.testing.assert_array_equal(rs.cpu().numpy(), o["recv_src_idx"])   # the dropped rows stay -1
    assert (rs.cpu().numpy()[dropped] == -1).all()


def test_two_stage_dispatch_with_node_rows_below_minus_one():
    from gpu_path import B, bf16_bits, to_dev, x_tensor
    T, H, E, K, R, rpn = 256, 1024, 64, 6, 8, 4
    d = make_inputs(T, H, E, K, R, seed=31)
    idx, w = to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    lay = B.alloc_layout(T, E, R, rpn, node_rows=True)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, rpn), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, st, rpn)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    M = int(lay.node_offset[-1].item())
    N = lay.num_recv
    bad, read_as, _ = _plant(lay.node_row.cpu().numpy(), -6, seed=9)
    lay.node_row.copy_(torch.from_numpy(bad))
    node_x = torch.full((M, H), -5.0, dtype=torch.bfloat16, device="cuda")
    recv_x = torch.full((N, H), -3.0, dtype=torch.bfloat16, device="cuda")
    rs = torch.full((N,), -9, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_dispatch_hierarchical(x_tensor(d["x_bits"]), idx, w, E, R, rpn, lay, node_x, recv_x, status,
                               recv_src_idx=rs)
    torch.cuda.synchronize()
    _expect(B, status)
    dst = lay.dst_row.cpu().numpy()
    o = oracle.dispatch_hierarchical(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, rpn, read_as, dst, M, N)
    # the rank rows reached through a node row the product reads as present
    node_of = np.arange(R) // rpn
    written = [dst[t, r] for t in range(T) for r in range(R) if dst[t, r] >= 0 and read_as[t, node_of[r]] >= 0]
    written = np.array(sorted(written))
    assert len(written) < N                    # some rows were dropped with their node row
    got = bf16_bits(recv_x).view(np.uint8).reshape(N, 2 * H)
    np.testing.assert_array_equal(got[written], o["recv_x"][written])
    np.testing.assert_array_equal(rs.cpu().numpy()[written], o["recv_src_idx"][written])
