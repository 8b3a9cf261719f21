"""Pins for the oracle's hierarchical (two-stage) path (no GPU).

* fp64 -> bf16 rounding: hand-worked ties, a value that double rounding
  through fp32 would get wrong, agreement with the fp32 -> bf16 routine and
  with torch's bf16 cast on fp32-representable values, bf16 subnormals;
* node rows against a numpy brute force (sorted token sets per node), and
  their counts against the layout's per-node counts;
* two-stage dispatch: node rows carry their source row (or its FP8 cast), and
  the receive buffers equal the single-stage dispatch bit for bit (bf16, FP8,
  row- and column-major scales);
* two-stage combine: the unweighted identity closed form
  out[t] = sum_n bf16(c_n(t) * x[t]) (torch's bf16 cast); one rank per node
  reduces to the single-stage combine exactly; one node to its bf16 rounding;
  weighted cases within half a bf16 ulp per node partial of the single-stage
  combine;
* capacity flags.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import make_inputs, make_rows


def test_double_to_bf16_hand_worked():
    v = [1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -40, -2.5, 0.0, -0.0, 255.5, 2 ** -130,
         3 * 2 ** -134]
    # 255.5: quantum 1 in [128, 256), a tie -> 256 (even); bf16 subnormals have
    # the fixed quantum 2^-133: 2^-130 = 8 quanta, 3 * 2^-134 = 1.5 quanta -> 2 (even)
    want = [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000, 0x8000, 0x4380, 0x0008, 0x0002]
    np.testing.assert_array_equal(oracle.double_to_bf16(v), np.array(want, np.uint16))
    # the same tie one fp32-invisible bit above rounds up (double rounding through fp32 would not)
    assert oracle.float_to_bf16([np.float32(1 + 2 ** -8 + 2 ** -40)])[0] == 0x3F80


def test_double_to_bf16_matches_float_paths():
    rng = np.random.Generator(np.random.PCG64(5))
    f = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    got = oracle.double_to_bf16(f.astype(np.float64))
    np.testing.assert_array_equal(got, oracle.float_to_bf16(f))
    tb = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, tb)


@pytest.mark.parametrize("T,K,E,R,rpn,mode", [
    (300, 8, 256, 64, 8, "uniform"), (200, 6, 64, 16, 4, "masked"), (128, 4, 16, 4, 1, "uniform"),
    (150, 8, 64, 8, 8, "uniform"), (97, 5, 96, 12, 3, "invalid"), (1, 8, 256, 8, 2, "uniform"),
])
def test_node_rows_brute_force(T, K, E, R, rpn, mode):
    rng = np.random.Generator(np.random.PCG64(T + R))
    if mode == "invalid":
        idx = rng.integers(-3, E + 3, size=(T, K)).astype(np.int64)
    else:
        idx = make_inputs(T, 8, E, K, R, seed=T, mask_frac=0.2 if mode == "masked" else 0.0,
                          with_x=False)["topk_idx"]
    off, rows, st = oracle.node_rows(idx, E, R, rpn)
    nodes = R // rpn
    el = E // R
    base = 0
    for n in range(nodes):
        toks = sorted({t for t in range(T) for e in idx[t] if 0 <= e < E and (e // el) // rpn == n})
        assert off[n] == base
        want = np.full(T, -1)
        want[toks] = base + np.arange(len(toks))
        np.testing.assert_array_equal(rows[:, n], want)
        base += len(toks)
    assert off[nodes] == base
    assert bool(st & oracle.EP_ERR_INVALID_INDEX) == (mode == "invalid" and bool(((idx < -1) | (idx >= E)).any()))
    if mode != "invalid":
        L = oracle.layout(idx, E, R, ranks_per_node=rpn)
        np.testing.assert_array_equal(np.diff(off), L.num_tokens_per_node)


def _case(T, H, E, K, R, rpn, seed, mask=0.0):
    d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=mask)
    L = oracle.layout(d["topk_idx"], E, R)
    off, rows, _ = oracle.node_rows(d["topk_idx"], E, R, rpn)
    return d, L, off, rows


@pytest.mark.parametrize("fp8,col", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("T,H,E,K,R,rpn", [(200, 256, 64, 6, 16, 4), (150, 128, 256, 8, 8, 8), (64, 384, 32, 4, 8, 1)])
def test_dispatch_two_stage_equals_single_stage(fp8, col, T, H, E, K, R, rpn):
    d, L, off, rows = _case(T, H, E, K, R, rpn, seed=T + H, mask=0.05)
    N, M = L.num_recv, int(off[-1])
    stride = (N + 3) // 4 * 4
    two = oracle.dispatch_hierarchical(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, rpn, rows, L.dst_row,
                                       M, N, fp8=fp8, sf_col_major=col, sf_stride=stride)
    one = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, capacity=N, fp8=fp8,
                          sf_col_major=col, sf_stride=stride)
    assert two["status"] == 0 and one["status"] == 0
    for k in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_idx") + (("recv_sf",) if fp8 else ()):
        np.testing.assert_array_equal(two[k], one[k], err_msg=k)
    # node buffers: every node row holds its source row (or its cast), rows of node n ascending in t
    src = two["node_src_idx"]
    assert (src >= 0).all()
    for n in range(len(off) - 1):
        assert (np.diff(src[off[n]:off[n + 1]]) > 0).all()
    if fp8:
        for j in range(0, M, max(1, M // 40)):
            q, sf = oracle.fp8_cast_row(d["x_bits"][src[j]])
            np.testing.assert_array_equal(two["node_x"][j], q)
            np.testing.assert_array_equal(two["node_sf"][j], sf)
    else:
        np.testing.assert_array_equal(two["node_x"].view(np.uint16), d["x_bits"][src])


def test_combine_two_stage_identity_closed_form():
    T, H, E, K, R, rpn = 200, 256, 64, 8, 16, 4
    d, L, off, rows = _case(T, H, E, K, R, rpn, seed=21, mask=0.1)
    res = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row)
    y = res["recv_x"].view(np.uint16)
    node_y, out, st = oracle.combine_hierarchical(y, d["topk_idx"], None, E, R, rpn, rows, L.dst_row, int(off[-1]))
    assert st == 0
    x = torch.from_numpy(d["x_bits"].view(np.int16)).view(torch.bfloat16).float()
    c = torch.from_numpy(L.is_token_in_rank.reshape(T, R // rpn, rpn).sum(axis=2).astype(np.float32))
    parts = (c[:, :, None] * x[:, None, :]).to(torch.bfloat16).double()      # [T, nodes, H]
    np.testing.assert_array_equal(out, parts.sum(dim=1).numpy())
    # node partials are bf16(c_n * x) of their token
    src_t, src_n = np.nonzero(rows >= 0)
    want = parts[src_t, src_n].float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(node_y[rows[src_t, src_n]], want)


@pytest.mark.parametrize("weighted", [False, True])
def test_combine_two_stage_special_cases(weighted):
    T, H, E, K, R = 150, 128, 64, 6, 8
    d, L, _, _ = _case(T, H, E, K, R, 1, seed=33, mask=0.05)
    y = make_rows(L.num_recv, H, seed=34)
    one, _ = oracle.combine(y, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, weighted=weighted)
    # one rank per node: unweighted partials are the rows themselves -> the same fp64 sum
    off1, rows1, _ = oracle.node_rows(d["topk_idx"], E, R, 1)
    _, out1, st = oracle.combine_hierarchical(y, d["topk_idx"], d["topk_weights"], E, R, 1, rows1, L.dst_row,
                                              int(off1[-1]), weighted=weighted)
    assert st == 0
    if not weighted:
        np.testing.assert_array_equal(out1, one)
    # one node: the single partial is the bf16 rounding of the whole sum
    offR, rowsR, _ = oracle.node_rows(d["topk_idx"], E, R, R)
    _, outR, _ = oracle.combine_hierarchical(y, d["topk_idx"], d["topk_weights"], E, R, R, rowsR, L.dst_row,
                                             int(offR[-1]), weighted=weighted)
    np.testing.assert_array_equal(oracle.double_to_bf16(outR), oracle.double_to_bf16(one))
    np.testing.assert_array_equal(outR, oracle.bf16_to_float(oracle.double_to_bf16(one)).reshape(outR.shape))
    # general nodes: each partial is off by at most half a bf16 ulp of itself
    off4, rows4, _ = oracle.node_rows(d["topk_idx"], E, R, 4)
    node_y, out4, _ = oracle.combine_hierarchical(y, d["topk_idx"], d["topk_weights"], E, R, 4, rows4, L.dst_row,
                                                  int(off4[-1]), weighted=weighted)
    py = np.abs(oracle.bf16_to_float(node_y).astype(np.float64))
    half_ulp = np.ldexp(1.0, np.frexp(py)[1] - 9)          # 2^(e-9) for |p| in [2^(e-1), 2^e)
    bound = np.zeros_like(out4)
    for n in range(rows4.shape[1]):
        j = rows4[:, n]
        bound += np.where(j[:, None] >= 0, half_ulp[np.maximum(j, 0)], 0.0)
    assert (np.abs(out4 - one) <= bound + 1e-300).all()


def test_hierarchical_capacity_flags():
    T, H, E, K, R, rpn = 64, 128, 16, 4, 8, 2
    d, L, off, rows = _case(T, H, E, K, R, rpn, seed=7)
    M = int(off[-1])
    res = oracle.dispatch_hierarchical(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, rpn, rows, L.dst_row,
                                       M - 3, L.num_recv)
    assert res["status"] & oracle.EP_ERR_CAPACITY
    y = make_rows(L.num_recv, H, seed=8)
    _, _, st = oracle.combine_hierarchical(y, d["topk_idx"], None, E, R, rpn, rows, L.dst_row, M - 1)
    assert st & oracle.EP_ERR_CAPACITY
