"""GPU parity of the hierarchical (two-stage) path against the CPU oracle.

* node rows and offsets bit-exact (masked, invalid, duplicate entries, one rank
  per node, one node, the node-limited large workload at full size), with the
  rest of the layout unchanged;
* two-stage dispatch: node buffers bit-exact against the oracle's two-stage
  dispatch, receive buffers bit-exact against the oracle's single-stage
  dispatch (bf16, FP8 with row- and column-major scales), and at full size
  identical to the GPU's single-stage dispatch;
* two-stage combine: node partials and outputs within the combine tolerance of
  the oracle; the unweighted identity closed form exact at full size; one rank
  per node identical to the single-stage combine;
* capacity overflow of the node buffers sets the status.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import make_config, make_inputs, make_rows

pytestmark = pytest.mark.gpu


def _layout(idx_np, E, R, rpn):
    from gpu_path import B, to_dev
    idx = to_dev(idx_np)
    T, K = idx.shape
    lay = B.alloc_layout(T, E, R, rpn, node_rows=True)
    lay.node_row.fill_(-7)
    lay.node_offset.fill_(-7)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, rpn), dtype=torch.uint8, device="cuda")
    ws.fill_(0x5A)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, st, rpn)
    return idx, lay, st


@pytest.mark.parametrize("T,K,E,R,rpn,mode", [
    (300, 8, 256, 64, 8, "uniform"), (777, 6, 96, 12, 3, "replace"), (513, 5, 40, 8, 2, "invalid"),
    (1000, 8, 256, 8, 1, "masked"), (200, 8, 256, 16, 16, "uniform"), (1, 4, 16, 4, 2, "uniform"),
    (300, 32, 2048, 1024, 32, "uniform"), (1024, 8, 256, 32, 1, "masked"),
])
def test_node_rows(T, K, E, R, rpn, mode):
    rng = np.random.Generator(np.random.PCG64(T + K + R))
    if mode in ("uniform", "masked"):
        idx = make_inputs(T, 8, E, K, R, seed=T, mask_frac=0.2 if mode == "masked" else 0.0,
                          with_x=False)["topk_idx"]
    elif mode == "replace":
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int64)
    else:
        idx = rng.integers(-3, E + 3, size=(T, K)).astype(np.int64)
    _, lay, st = _layout(idx, E, R, rpn)
    off, rows, ost = oracle.node_rows(idx, E, R, rpn)
    np.testing.assert_array_equal(lay.node_row.cpu().numpy(), rows)
    np.testing.assert_array_equal(lay.node_offset.cpu().numpy(), off)
    L = oracle.layout(idx, E, R, ranks_per_node=rpn)
    np.testing.assert_array_equal(lay.num_tokens_per_node.cpu().numpy(), L.num_tokens_per_node)
    np.testing.assert_array_equal(lay.dst_row.cpu().numpy(), L.dst_row)
    np.testing.assert_array_equal(lay.rank_offset.cpu().numpy(), L.rank_offset)
    assert int(st.item()) == (ost | L.status)


def _dispatch(B, x, idx, w, E, R, rpn, lay, M, N, fp8, col):
    T, H = x.shape
    K = idx.shape[1]
    nb = H // 128
    if fp8:
        node_x = torch.full((M, H), 0x33, dtype=torch.uint8, device="cuda")
        node_sf = torch.full((M * nb,), -2.0, dtype=torch.float32, device="cuda")
        recv_x = torch.full((N, H), 0x55, dtype=torch.uint8, device="cuda")
        stride = (N + 3) // 4 * 4
        recv_sf = torch.full(((nb * stride) if col else N * nb,), -1.0, dtype=torch.float32, device="cuda")
    else:
        node_x = torch.full((M, H), -5.0, dtype=torch.bfloat16, device="cuda")
        node_sf = recv_sf = None
        recv_x = torch.full((N, H), -3.0, dtype=torch.bfloat16, device="cuda")
    node_src = torch.full((M,), -9, dtype=torch.int32, device="cuda")
    ri = torch.full((N, K), -9, dtype=torch.int32, device="cuda")
    rw = torch.full((N, K), -9.0, dtype=torch.float32, device="cuda")
    rs = torch.full((N,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_dispatch_hierarchical(x, idx, w, E, R, rpn, lay, node_x, recv_x, st, node_sf=node_sf, node_src_idx=node_src,
                               recv_sf=recv_sf, recv_topk_idx=ri, recv_topk_weights=rw, recv_src_idx=rs,
                               out_dtype=B.EP_FP8_E4M3 if fp8 else B.EP_BF16, sf_col_major=col)
    torch.cuda.synchronize()
    return dict(node_x=node_x, node_sf=node_sf, node_src_idx=node_src, recv_x=recv_x, recv_sf=recv_sf,
                recv_topk_idx=ri, recv_topk_weights=rw, recv_src_idx=rs, status=st)


def _bytes(t):
    from gpu_path import bf16_bits
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return bf16_bits(t).view(np.uint8).reshape(t.shape[0], 2 * t.shape[1])


@pytest.mark.parametrize("fp8,col", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("T,H,E,K,R,rpn,mask", [
    (500, 1024, 64, 6, 16, 4, 0.1), (300, 7168, 256, 8, 64, 8, 0.0), (77, 256, 32, 4, 8, 1, 0.0),
    (200, 512, 2048, 32, 1024, 32, 0.1), (33, 4096, 128, 8, 8, 8, 0.05),
])
def test_dispatch_hierarchical(fp8, col, T, H, E, K, R, rpn, mask):
    _check_dispatch_hierarchical(fp8, col, T, H, E, K, R, rpn, mask, seed=T + H + R)


def _check_dispatch_hierarchical(fp8, col, T, H, E, K, R, rpn, mask, seed):
    from gpu_path import B, x_tensor
    d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=mask)
    idx, lay, _ = _layout(d["topk_idx"], E, R, rpn)
    w = torch.from_numpy(d["topk_weights"]).cuda()
    N, M = lay.num_recv, int(lay.node_offset[-1].item())
    g = _dispatch(B, x_tensor(d["x_bits"]), idx, w, E, R, rpn, lay, M, N, fp8, col)
    assert int(g["status"].item()) == 0
    L = oracle.layout(d["topk_idx"], E, R)
    _, rows, _ = oracle.node_rows(d["topk_idx"], E, R, rpn)
    stride = (N + 3) // 4 * 4
    two = oracle.dispatch_hierarchical(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, rpn, rows, L.dst_row,
                                       M, N, fp8=fp8, sf_col_major=col, sf_stride=stride)
    np.testing.assert_array_equal(_bytes(g["node_x"]), two["node_x"])
    np.testing.assert_array_equal(g["node_src_idx"].cpu().numpy(), two["node_src_idx"])
    one = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, capacity=N, fp8=fp8,
                          sf_col_major=col, sf_stride=stride)
    np.testing.assert_array_equal(_bytes(g["recv_x"]), one["recv_x"])
    for k in ("recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(g[k].cpu().numpy(), one[k], err_msg=k)
    if fp8:
        np.testing.assert_array_equal(g["node_sf"].cpu().numpy().reshape(M, H // 128), two["node_sf"])
        if col:
            nb = H // 128
            got = g["recv_sf"].cpu().numpy()[:nb * stride].reshape(nb, stride)[:, :N]
            want = one["recv_sf"][:nb * stride].reshape(nb, stride)[:, :N]
        else:
            got, want = g["recv_sf"].cpu().numpy().reshape(N, H // 128), one["recv_sf"]
        np.testing.assert_array_equal(got, want)


def test_dispatch_hierarchical_full_size_matches_single_stage():
    """The node-limited large workload (T=32768, R=64, 8 ranks per node):
    node rows against the oracle, every received row and its metadata
    identical to the single-stage dispatch on the GPU."""
    from gpu_path import B, run_dispatch, x_tensor
    d = make_config("large")
    c = d["cfg"]
    idx, lay, st = _layout(d["topk_idx"], c.E, c.R, c.ranks_per_node)
    off, rows, _ = oracle.node_rows(d["topk_idx"], c.E, c.R, c.ranks_per_node)
    np.testing.assert_array_equal(lay.node_row.cpu().numpy(), rows)
    x = x_tensor(d["x_bits"])
    w = torch.from_numpy(d["topk_weights"]).cuda()
    N, M = lay.num_recv, int(off[-1])
    g = _dispatch(B, x, idx, w, c.E, c.R, c.ranks_per_node, lay, M, N, False, False)
    assert int(g["status"].item()) == 0
    ref = run_dispatch(x, idx, w, c.E, c.R, lay, N)
    torch.cuda.synchronize()
    for k in ("recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        assert torch.equal(g[k], ref[k]), k
    assert torch.equal(g["recv_x"].view(torch.int16), ref["recv_x"].view(torch.int16))
    src = g["node_src_idx"].long()
    assert torch.equal(g["node_x"].view(torch.int16), x.view(torch.int16)[src])
    np.testing.assert_array_equal(g["node_src_idx"].cpu().numpy(),
                                  np.concatenate([np.flatnonzero(rows[:, n] >= 0) for n in range(rows.shape[1])]))


def _combine(B, y, idx, w, E, R, rpn, lay, M, T, H):
    node_y = torch.full((M, H), 9.0, dtype=torch.bfloat16, device="cuda")
    out = torch.full((T, H), 5.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_combine_hierarchical(y, idx, w, E, R, rpn, lay, node_y, out, st)
    torch.cuda.synchronize()
    return node_y, out, st


@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("T,H,E,K,R,rpn,mask", [
    (500, 1024, 64, 6, 16, 4, 0.1), (300, 7168, 256, 8, 64, 8, 0.0), (200, 256, 2048, 32, 1024, 32, 0.1),
    (64, 512, 32, 4, 8, 8, 0.0),
])
def test_combine_hierarchical(weighted, T, H, E, K, R, rpn, mask):
    _check_combine_hierarchical(weighted, T, H, E, K, R, rpn, mask, seed=T + 3 * H)


def _check_combine_hierarchical(weighted, T, H, E, K, R, rpn, mask, seed):
    from gpu_path import B, bf16_bits, x_tensor
    d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=mask, with_x=False)
    idx, lay, _ = _layout(d["topk_idx"], E, R, rpn)
    w = torch.from_numpy(d["topk_weights"]).cuda()
    N, M = lay.num_recv, int(lay.node_offset[-1].item())
    y_bits = make_rows(N, H, seed=T + 5)
    node_y, out, st = _combine(B, x_tensor(y_bits), idx, w if weighted else None, E, R, rpn, lay, M, T, H)
    assert int(st.item()) == 0
    L = oracle.layout(d["topk_idx"], E, R)
    _, rows, _ = oracle.node_rows(d["topk_idx"], E, R, rpn)
    ony, oout, _ = oracle.combine_hierarchical(y_bits, d["topk_idx"], d["topk_weights"], E, R, rpn, rows, L.dst_row,
                                               M, weighted=weighted)
    yf = oracle.bf16_to_float(y_bits).astype(np.float64)
    # |c| * |y| summed per (token, node) and per token: the tolerance scale
    el = E // R
    coef = np.zeros((T, R))
    tt, rr = np.nonzero(L.dst_row >= 0)
    if weighted:
        for k in range(K):
            e = d["topk_idx"][:, k]
            ok = e >= 0
            np.add.at(coef, (np.flatnonzero(ok), e[ok] // el), np.abs(d["topk_weights"][ok, k]))
    else:
        coef[tt, rr] = 1.0
    scale_node = np.zeros((M, H))
    scale_tok = np.zeros((T, H))
    n_node = np.zeros(M)
    for t, r in zip(tt, rr):
        a = coef[t, r] * np.abs(yf[L.dst_row[t, r]])
        scale_node[rows[t, r // rpn]] += a
        scale_tok[t] += a
        n_node[rows[t, r // rpn]] += 1
    g_node = oracle.bf16_to_float(bf16_bits(node_y).reshape(M, H)).astype(np.float64)
    want_node = oracle.bf16_to_float(ony).astype(np.float64)
    assert (np.abs(g_node - want_node) <= 1e-2 * scale_node).all()
    _check_two_stage_tight(g_node, want_node, n_node, scale_node, K if weighted else 0, rows, bf16_bits(out), T, H)
    g_out = oracle.bf16_to_float(bf16_bits(out).reshape(T, H)).astype(np.float64)
    assert (np.abs(g_out - oout) <= 1e-2 * scale_tok).all()
    empty = L.is_token_in_rank.sum(axis=1) == 0
    assert (g_out[empty] == 0).all()


def _check_two_stage_tight(g_node, want_node, n_node, scale_node, m, node_rows, out_bits, T, H):
    """fp32-accumulation bounds of both stages (tests/tolerance.py).
    Stage 1: the GPU's node partial bf16(P32) and the oracle's bf16(P) are
    each within 2^-8 |P| (+ the fp32 error of P32) of the exact partial P,
    and |P| <= |bf16(P)| / (1 - 2^-8).  Stage 2: the output is bf16 of the
    fp32 sum of the GPU's own node partials."""
    from tolerance import BF16_MIN_SUBNORMAL, U32, U_BF16, bf16_bits_to_f64, sum_bound
    p_abs = np.abs(want_node) / (1.0 - U_BF16)
    tight_node = (2.0 * U_BF16 * p_abs + 2.0 * (n_node[:, None] + m + 1) * U32 * scale_node
                  + 2.0 * BF16_MIN_SUBNORMAL)
    assert (np.abs(g_node - want_node) <= tight_node).all()
    exact = np.zeros((T, H))
    mag = np.zeros((T, H))
    n_parts = np.zeros(T)
    for n in range(node_rows.shape[1]):
        ok = node_rows[:, n] >= 0
        part = g_node[node_rows[ok, n]]
        exact[ok] += part
        mag[ok] += np.abs(part)
        n_parts += ok
    g_out = bf16_bits_to_f64(out_bits.reshape(T, H))
    assert (np.abs(g_out - exact) <= sum_bound(exact, mag, n_parts)).all()


def test_combine_hierarchical_identity_full_size():
    """Dispatch -> identity -> two-stage combine on the large workload:
    out[t] = bf16(sum over nodes n of bf16(c_n(t) * x[t])) exactly."""
    from gpu_path import B, run_dispatch, x_tensor
    d = make_config("large")
    c = d["cfg"]
    idx, lay, _ = _layout(d["topk_idx"], c.E, c.R, c.ranks_per_node)
    x = x_tensor(d["x_bits"])
    w = torch.from_numpy(d["topk_weights"]).cuda()
    N, M = lay.num_recv, int(lay.node_offset[-1].item())
    res = run_dispatch(x, idx, w, c.E, c.R, lay, N, with_meta=False)
    node_y, out, st = _combine(B, res["recv_x"], idx, None, c.E, c.R, c.ranks_per_node, lay, M, c.T, c.H)
    assert int(st.item()) == 0
    nodes = c.R // c.ranks_per_node
    cn = lay.is_token_in_rank.view(c.T, nodes, c.ranks_per_node).sum(dim=2).float()     # [T, nodes]
    want = torch.zeros((c.T, c.H), dtype=torch.float32, device="cuda")
    for n in range(nodes):
        want += (cn[:, n:n + 1] * x.float()).to(torch.bfloat16).float()
    assert torch.equal(out.float(), want.to(torch.bfloat16).float())


def test_combine_hierarchical_one_rank_per_node_equals_single_stage():
    from gpu_path import B, run_combine, x_tensor
    T, H, E, K, R = 700, 2048, 64, 6, 16
    d = make_inputs(T, H, E, K, R, seed=9, mask_frac=0.05, with_x=False)
    idx, lay, _ = _layout(d["topk_idx"], E, R, 1)
    N, M = lay.num_recv, int(lay.node_offset[-1].item())
    y = x_tensor(make_rows(N, H, seed=10))
    _, out, st = _combine(B, y, idx, None, E, R, 1, lay, M, T, H)
    ref, _ = run_combine(y, idx, None, E, R, lay, T, H)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_hierarchical_node_capacity_overflow():
    from gpu_path import B, x_tensor
    T, H, E, K, R, rpn = 400, 512, 64, 4, 8, 2
    d = make_inputs(T, H, E, K, R, seed=12)
    idx, lay, _ = _layout(d["topk_idx"], E, R, rpn)
    w = torch.from_numpy(d["topk_weights"]).cuda()
    N, M = lay.num_recv, int(lay.node_offset[-1].item())
    g = _dispatch(B, x_tensor(d["x_bits"]), idx, w, E, R, rpn, lay, M - 10, N, False, False)
    assert int(g["status"].item()) & oracle.EP_ERR_CAPACITY
    _, _, st = _combine(B, g["recv_x"], idx, None, E, R, rpn, lay, M - 10, T, H)
    assert int(st.item()) & oracle.EP_ERR_CAPACITY


@pytest.mark.parametrize("weighted", [False, True])
def test_combine_hierarchical_short_y(weighted):
    """Expert rows beyond num_y_rows are skipped: each node partial is the sum
    of the node's remaining rows (zero when none remain), as in the oracle;
    the capacity bit is set."""
    from gpu_path import B, bf16_bits, x_tensor
    T, H, E, K, R, rpn = 400, 512, 64, 6, 16, 4
    d = make_inputs(T, H, E, K, R, seed=31, mask_frac=0.05, with_x=False)
    idx, lay, _ = _layout(d["topk_idx"], E, R, rpn)
    w = torch.from_numpy(d["topk_weights"]).cuda()
    N, M = lay.num_recv, int(lay.node_offset[-1].item())
    n_y = N - 300
    y_bits = make_rows(n_y, H, seed=32)
    node_y, out, st = _combine(B, x_tensor(y_bits), idx, w if weighted else None, E, R, rpn, lay, M, T, H)
    assert int(st.item()) & oracle.EP_ERR_CAPACITY
    L = oracle.layout(d["topk_idx"], E, R)
    _, rows, _ = oracle.node_rows(d["topk_idx"], E, R, rpn)
    ony, oout, ost = oracle.combine_hierarchical(y_bits, d["topk_idx"], d["topk_weights"], E, R, rpn, rows,
                                                 L.dst_row, M, weighted=weighted)
    assert ost & oracle.EP_ERR_CAPACITY
    yf = oracle.bf16_to_float(y_bits).astype(np.float64)
    el = E // R
    scale_node = np.zeros((M, H))
    scale_tok = np.zeros((T, H))
    n_node = np.zeros(M)
    tt, rr = np.nonzero((L.dst_row >= 0) & (L.dst_row < n_y))
    for t, r in zip(tt, rr):
        c = 1.0
        if weighted:
            c = sum(abs(float(d["topk_weights"][t, k])) for k in range(K)
                    if d["topk_idx"][t, k] >= 0 and d["topk_idx"][t, k] // el == r)
        a = c * np.abs(yf[L.dst_row[t, r]])
        scale_node[rows[t, r // rpn]] += a
        scale_tok[t] += a
        n_node[rows[t, r // rpn]] += 1
    g_node = oracle.bf16_to_float(bf16_bits(node_y).reshape(M, H)).astype(np.float64)
    want_node = oracle.bf16_to_float(ony).astype(np.float64)
    assert (np.abs(g_node - want_node) <= 1e-2 * scale_node).all()
    _check_two_stage_tight(g_node, want_node, n_node, scale_node, K if weighted else 0, rows, bf16_bits(out), T, H)
    g_out = oracle.bf16_to_float(bf16_bits(out).reshape(T, H)).astype(np.float64)
    assert (np.abs(g_out - oout) <= 1e-2 * scale_tok).all()


@pytest.mark.parametrize("i", range(24))
def test_random_hierarchical(i):
    """Two-stage dispatch and combine on the random sweep's shapes (node
    groups of the case, else a middle divisor of R): node buffers and receive
    buffers exact, combine within tolerance."""
    from test_gpu_random import _draw_case
    c = _draw_case(i)
    R = c["R"]
    divisors = [d for d in range(1, R + 1) if R % d == 0]
    rpn = c["rpn"] or divisors[len(divisors) // 2]
    _check_dispatch_hierarchical(c["fp8"], c["fp8"] and i % 2 == 1, c["T"], c["H"], c["E"], c["K"], R, rpn, c["mask"],
                                 seed=c["seed"])
    _check_combine_hierarchical(c["weighted"], c["T"], c["H"], c["E"], c["K"], R, rpn, c["mask"], seed=c["seed"] + 7)

