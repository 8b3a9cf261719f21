"""Pins for the CPU oracle's dispatch and combine (no GPU).

* the hand-worked example's received metadata;
* every received row equals its source row byte for byte, and the received
  metadata follows an independent per-(row, k) numpy formulation;
* compact (sampled) dispatch equals the full dispatch at the same rows;
* closed forms of dispatch -> identity expert -> combine:
  unweighted out[t] = n(t) * x[t] exactly, weighted out[t] = x[t] * sum of
  t's unmasked weights;
* combine of arbitrary expert rows against an independent scatter-add
  formulation (``np.add.at``);
* capacity and invalid-index status bits.
"""
import json
import os

import numpy as np
import pytest

import oracle
from combine_ep_get_gb300.inputs import make_inputs, make_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(T, H, E, K, R, seed, mask=0.0):
    d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=mask)
    L = oracle.layout(d["topk_idx"], E, R)
    return d, L


def test_handworked_dispatch_metadata_and_combine():
    g = json.load(open(os.path.join(GOLDEN, "layout_handworked.json")))
    idx = np.array(g["topk_idx"], np.int64)
    w = np.array(g["topk_weights"], np.float32)
    E, R = g["E"], g["R"]
    T, H = idx.shape[0], 128
    x = make_rows(T, H, seed=5)
    L = oracle.layout(idx, E, R)
    res = oracle.dispatch(x, idx, w, E, R, L.dst_row)
    np.testing.assert_array_equal(res["recv_src_idx"], g["recv_src_idx"])
    np.testing.assert_array_equal(res["recv_topk_idx"], g["recv_topk_idx"])
    np.testing.assert_array_equal(res["recv_topk_weights"], np.array(g["recv_topk_weights"], np.float32))
    # weighted combine of the identity expert: x[t] * sum_r c(t, r)
    y = res["recv_x"].view(np.uint16)
    out, st = oracle.combine(y, idx, w, E, R, L.dst_row, weighted=True)
    coef = np.array(g["combine_coef_per_token_rank"]).sum(axis=1)
    np.testing.assert_allclose(out, coef[:, None] * oracle.bf16_to_float(x), rtol=0, atol=0)


@pytest.mark.parametrize("T,H,E,K,R,mask", [(128, 256, 16, 4, 4, 0.0), (200, 384, 64, 8, 8, 0.1),
                                            (61, 128, 32, 3, 16, 0.0)])
def test_dispatch_rows_and_metadata(T, H, E, K, R, mask):
    d, L = _case(T, H, E, K, R, seed=T + H, mask=mask)
    res = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row)
    N = L.num_recv
    assert res["recv_x"].shape[0] == N and res["status"] == 0
    src = res["recv_src_idx"]
    # payload: byte-identical to the source row
    np.testing.assert_array_equal(res["recv_x"].view(np.uint16), d["x_bits"][src])
    # destination row of (src, r) is this row, for exactly one r
    rows = np.arange(N)
    hit = (L.dst_row[src] == rows[:, None])
    assert (hit.sum(axis=1) == 1).all()
    rank = hit.argmax(axis=1)
    # metadata by an independent formulation over (row, k)
    el = E // R
    e = d["topk_idx"][src]                                       # [N, K]
    on = (e >= 0) & (e // el == rank[:, None])
    np.testing.assert_array_equal(res["recv_topk_idx"], np.where(on, e - rank[:, None] * el, -1))
    np.testing.assert_array_equal(res["recv_topk_weights"], np.where(on, d["topk_weights"][src], 0.0))
    # receive order inside a rank is ascending source token
    for r in range(R):
        s = src[L.rank_offset[r]:L.rank_offset[r + 1]]
        assert (np.diff(s) > 0).all()


def test_compact_dispatch_matches_full():
    d, L = _case(96, 256, 32, 6, 8, seed=11, mask=0.05)
    full = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], 32, 8, L.dst_row)
    toks = np.array([0, 5, 17, 95, 42], np.int32)
    part = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], 32, 8, L.dst_row, tokens=toks)
    rows = part["rows"]
    assert len(rows) == int((L.dst_row[toks] >= 0).sum())
    for key in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(part[key], full[key][rows], err_msg=key)


@pytest.mark.parametrize("T,H,E,K,R,mask", [(128, 256, 16, 4, 4, 0.0), (300, 512, 256, 8, 64, 0.05)])
def test_round_trip_closed_form(T, H, E, K, R, mask):
    d, L = _case(T, H, E, K, R, seed=3 * T, mask=mask)
    res = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row)
    y = res["recv_x"].view(np.uint16)
    x = oracle.bf16_to_float(d["x_bits"]).astype(np.float64)
    n_t = L.is_token_in_rank.sum(axis=1)
    out, st = oracle.combine(y, d["topk_idx"], None, E, R, L.dst_row, weighted=False)
    assert st == 0
    np.testing.assert_array_equal(out, n_t[:, None] * x)
    outw, _ = oracle.combine(y, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, weighted=True)
    wsum = np.where(d["topk_idx"] >= 0, d["topk_weights"].astype(np.float64), 0.0).sum(axis=1)
    np.testing.assert_allclose(outw, wsum[:, None] * x, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("weighted", [False, True])
def test_combine_against_scatter_add(weighted):
    T, H, E, K, R = 150, 256, 64, 6, 8
    d, L = _case(T, H, E, K, R, seed=77, mask=0.1)
    N = L.num_recv
    y = make_rows(N, H, seed=78)
    yf = oracle.bf16_to_float(y).astype(np.float64)
    el = E // R
    ref = np.zeros((T, H))
    for k in range(K):
        e = d["topk_idx"][:, k]
        ok = e >= 0
        t = np.flatnonzero(ok)
        r = e[ok] // el
        rows = L.dst_row[t, r]
        c = d["topk_weights"][t, k].astype(np.float64) if weighted else None
        if weighted:
            np.add.at(ref, t, c[:, None] * yf[rows])
    if not weighted:
        tt, rr = np.nonzero(L.dst_row >= 0)
        np.add.at(ref, tt, yf[L.dst_row[tt, rr]])
    out, st = oracle.combine(y, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, weighted=weighted)
    assert st == 0
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_sampled_combine_matches_full():
    d, L = _case(64, 128, 16, 4, 4, seed=5)
    y = make_rows(L.num_recv, 128, seed=6)
    full, _ = oracle.combine(y, d["topk_idx"], d["topk_weights"], 16, 4, L.dst_row, weighted=True)
    toks = np.array([3, 0, 63], np.int32)
    part, _ = oracle.combine(y, d["topk_idx"], d["topk_weights"], 16, 4, L.dst_row, weighted=True,
                             tokens=toks)
    np.testing.assert_array_equal(part, full[toks])


def test_capacity_and_invalid_flags():
    d, L = _case(64, 128, 16, 4, 4, seed=9)
    res = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], 16, 4, L.dst_row,
                          capacity=L.num_recv - 3)
    assert res["status"] & oracle.EP_ERR_CAPACITY
    y = make_rows(L.num_recv - 3, 128, seed=1)
    _, st = oracle.combine(y, d["topk_idx"], None, 16, 4, L.dst_row)
    assert st & oracle.EP_ERR_CAPACITY
    bad = d["topk_idx"].copy()
    bad[3, 1] = 99
    L2 = oracle.layout(bad, 16, 4)
    assert L2.status & oracle.EP_ERR_INVALID_INDEX
    # the bad entry is skipped: token 3 keeps its other ranks
    good = bad.copy()
    good[3, 1] = -1
    L3 = oracle.layout(good, 16, 4)
    np.testing.assert_array_equal(L2.dst_row, L3.dst_row)


def test_combined_topk_weights_closed_form():
    """Each slot's weight travels only in the row of the rank holding its
    expert, so combining the received weight rows returns topk_weights
    exactly for valid slots and 0 for masked ones."""
    T, H, E, K, R = 300, 64, 64, 6, 8
    d, L = _case(T, H, E, K, R, seed=41, mask=0.15)
    res = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row)
    comb, st = oracle.combine_topk_weights(res["recv_topk_weights"], L.dst_row)
    assert st == 0
    want = np.where(d["topk_idx"] >= 0, d["topk_weights"], 0.0).astype(np.float32)
    np.testing.assert_array_equal(comb, want)
    # scaled received weights combine to the scaled weights
    comb2, _ = oracle.combine_topk_weights(res["recv_topk_weights"] * 2.0, L.dst_row)
    np.testing.assert_array_equal(comb2, 2.0 * want)
    # a short row count flags and skips
    _, st = oracle.combine_topk_weights(res["recv_topk_weights"][:L.num_recv - 5], L.dst_row)
    assert st & oracle.EP_ERR_CAPACITY


def test_expert_stats_accumulate():
    d, L = _case(64, 64, 16, 4, 4, seed=2)
    stats = np.zeros(16, np.int64)
    oracle.accumulate_expert_stats(L.num_tokens_per_expert, stats)
    oracle.accumulate_expert_stats(L.num_tokens_per_expert, stats)
    np.testing.assert_array_equal(stats, 2 * np.bincount(d["topk_idx"][d["topk_idx"] >= 0], minlength=16))


def test_openmp_build_gives_the_same_results():
    """The oracle's OpenMP build (token loops of dispatch and combine split
    over host threads, used for the all-cores CPU baseline) returns exactly
    what the single-threaded build returns."""
    T, H, E, K, R = 300, 512, 64, 6, 8
    d = make_inputs(T, H, E, K, R, seed=21, mask_frac=0.1)
    L = oracle.layout(d["topk_idx"], E, R)
    outs = []
    for parallel in (False, True):
        if parallel:
            with oracle.threads() as n:
                if n is None:
                    pytest.skip("no OpenMP build on this host")
                res = _dispatch_and_combine(d, E, R, L)
        else:
            res = _dispatch_and_combine(d, E, R, L)
        outs.append(res)
    for a, b in zip(outs[0], outs[1]):
        np.testing.assert_array_equal(a, b)


def _dispatch_and_combine(d, E, R, L):
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, capacity=L.num_recv)
    f = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, capacity=L.num_recv,
                        fp8=True)
    c, st = oracle.combine(o["recv_x"].view(np.uint16), d["topk_idx"], d["topk_weights"], E, R, L.dst_row,
                           weighted=True)
    return [o["recv_x"], o["recv_topk_idx"], o["recv_topk_weights"], o["recv_src_idx"], f["recv_x"], f["recv_sf"],
            c, np.array([o["status"], st])]
