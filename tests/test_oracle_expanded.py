"""Pins for the oracle's expanded (per-expert) receive layout, dispatch and
combine (no GPU): the hand-worked example, an independent stable-sort
formulation, block invariants, and the identity-expert closed forms."""
import json
import os

import numpy as np
import pytest

import oracle
from combine_ep_get_gb300.inputs import make_inputs, make_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_expanded(topk_idx, E, align):
    T, K = topk_idx.shape
    flat = topk_idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    order = np.flatnonzero(valid)
    # stable sort of the valid (t, k) entries by expert keeps (token, k) order
    srt = order[np.argsort(flat[order], kind="stable")]
    counts = np.bincount(flat[valid], minlength=E)
    starts = np.concatenate([[0], np.cumsum(-(-counts // align) * align)])
    rows = -np.ones(T * K, np.int64)
    pos_in_expert = np.zeros(E, np.int64)
    for i in srt:
        e = flat[i]
        rows[i] = starts[e] + pos_in_expert[e]
        pos_in_expert[e] += 1
    return rows.reshape(T, K)


def test_handworked():
    g = json.load(open(os.path.join(GOLDEN, "layout_handworked.json")))
    idx = np.array(g["topk_idx"], np.int64)
    L = oracle.layout(idx, g["E"], g["R"], g["ranks_per_node"], g["expert_alignment"])
    rows, st = oracle.expanded_rows(idx, g["E"], L.expert_offset)
    assert st == 0
    np.testing.assert_array_equal(rows, g["expanded_row"])


@pytest.mark.parametrize("T,K,E,R,align,mode", [
    (64, 4, 16, 4, 1, "uniform"), (300, 8, 256, 8, 128, "masked"), (257, 6, 48, 16, 7, "replace"),
    (96, 5, 40, 8, 3, "invalid"), (1, 1, 1, 1, 1, "uniform"),
])
def test_against_stable_sort(T, K, E, R, align, mode):
    rng = np.random.Generator(np.random.PCG64(T + K))
    if mode in ("uniform", "masked"):
        idx = make_inputs(T, 8, E, K, R, seed=T, mask_frac=0.2 if mode == "masked" else 0.0,
                          with_x=False)["topk_idx"]
    elif mode == "replace":
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int64)       # duplicates within a token
    else:
        idx = rng.integers(-3, E + 3, size=(T, K)).astype(np.int64)
    L = oracle.layout(idx, E, R, 0, align)
    rows, st = oracle.expanded_rows(idx, E, L.expert_offset)
    np.testing.assert_array_equal(rows, brute_expanded(idx, E, align))
    assert bool(st & oracle.EP_ERR_INVALID_INDEX) == (mode == "invalid")
    # block invariants: expert e's rows are expert_offset[e] + [0, count)
    v = rows >= 0
    for e in range(E):
        r = np.sort(rows[(idx == e) & v])
        np.testing.assert_array_equal(r, L.expert_offset[e] + np.arange(L.num_tokens_per_expert[e]))
    assert len(np.unique(rows[v])) == int(v.sum())


@pytest.mark.parametrize("weighted", [False, True])
def test_dispatch_and_combine_closed_forms(weighted):
    T, H, E, K, R = 200, 256, 64, 6, 8
    d = make_inputs(T, H, E, K, R, seed=5, mask_frac=0.1)
    L = oracle.layout(d["topk_idx"], E, R, 0, 16)
    rows, _ = oracle.expanded_rows(d["topk_idx"], E, L.expert_offset)
    cap = int(L.expert_offset[-1])
    res = oracle.dispatch_expanded(d["x_bits"], d["topk_weights"], rows, cap)
    assert res["status"] == 0
    t_of, k_of = np.nonzero(rows >= 0)
    r = rows[t_of, k_of]
    np.testing.assert_array_equal(res["recv_x"][r].view(np.uint16), d["x_bits"][t_of])
    np.testing.assert_array_equal(res["recv_src_idx"][r], t_of)
    np.testing.assert_array_equal(res["recv_weight"][r], d["topk_weights"][t_of, k_of])
    # padding rows are untouched
    pad = np.setdiff1d(np.arange(cap), r)
    assert (res["recv_src_idx"][pad] == -1).all()
    y = res["recv_x"].view(np.uint16)
    out, st = oracle.combine_expanded(y, d["topk_weights"], rows, weighted=weighted)
    x = oracle.bf16_to_float(d["x_bits"]).astype(np.float64)
    v = rows >= 0
    c = np.where(v, d["topk_weights"].astype(np.float64), 0.0).sum(axis=1) if weighted else v.sum(axis=1)
    np.testing.assert_allclose(out, c[:, None] * x, rtol=1e-12, atol=1e-12)


def test_combine_against_scatter_add():
    T, H, E, K, R = 150, 128, 32, 4, 4
    d = make_inputs(T, H, E, K, R, seed=8, mask_frac=0.15, with_x=False)
    L = oracle.layout(d["topk_idx"], E, R, 0, 4)
    rows, _ = oracle.expanded_rows(d["topk_idx"], E, L.expert_offset)
    y = make_rows(int(L.expert_offset[-1]), H, seed=9)
    yf = oracle.bf16_to_float(y).astype(np.float64)
    ref = np.zeros((T, H))
    t_of, k_of = np.nonzero(rows >= 0)
    np.add.at(ref, t_of, d["topk_weights"][t_of, k_of].astype(np.float64)[:, None] * yf[rows[t_of, k_of]])
    out, _ = oracle.combine_expanded(y, d["topk_weights"], rows, weighted=True)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("align", [1, 16])
def test_dispatch_fp8_col_major_scales_are_the_transpose(align):
    """Column-major FP8 scales of the expanded dispatch (the TMA-aligned
    scale layout a grouped GEMM loads): scale (row, b) sits at
    b * stride + row, with stride = capacity rounded up to 4.  Against the
    row-major result of the same call: every written row's scales are its
    row-major scales, and the entries of padding rows and of the stride's
    tail keep the fill value."""
    T, H, E, K, R = 90, 512, 32, 5, 4
    d = make_inputs(T, H, E, K, R, seed=11 + align, mask_frac=0.1)
    L = oracle.layout(d["topk_idx"], E, R, 0, align)
    rows, _ = oracle.expanded_rows(d["topk_idx"], E, L.expert_offset)
    cap = int(L.expert_offset[-1])
    stride = (cap + 3) // 4 * 4
    nb = H // 128
    rm = oracle.dispatch_expanded(d["x_bits"], d["topk_weights"], rows, cap, fp8=True)
    cm = oracle.dispatch_expanded(d["x_bits"], d["topk_weights"], rows, cap, fp8=True, sf_col_major=True,
                                  sf_stride=stride, sf_fill=-5.0)
    assert rm["status"] == 0 and cm["status"] == 0
    np.testing.assert_array_equal(cm["recv_x"], rm["recv_x"])
    written = np.unique(rows[rows >= 0])
    cols = cm["recv_sf"].reshape(nb, stride)
    np.testing.assert_array_equal(cols[:, written].T, rm["recv_sf"][written])
    unwritten = np.setdiff1d(np.arange(stride), written)
    if align > 1:
        assert len(unwritten) > stride - cap        # padding rows exist inside the columns
    assert (cols[:, unwritten] == -5.0).all()
    # the scales themselves follow the single-row cast
    for t in (0, T // 2, T - 1):
        for k in range(K):
            if rows[t, k] >= 0:
                _, sf = oracle.fp8_cast_row(d["x_bits"][t])
                np.testing.assert_array_equal(cols[:, rows[t, k]], sf)
