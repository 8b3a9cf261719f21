"""Pins for the CPU oracle's routing layout (no GPU).

* a hand-worked example (tests/golden/layout_handworked.json);
* brute force on small inputs by an independent numpy formulation that builds
  each rank's receive list by filtering and sorting (the oracle instead
  streams per-rank counters over tokens);
* the count invariants of "DeepEP Symmetric Memory" section 7.3 on all five
  workload shapes;
* the expected number of distinct groups per token, the closed form of the
  ``get_expected_topk`` helper inside ``get_theoretical_num_sms``
  ("DeepEP V2 ElasticBuffer architecture"), against the oracle's mean n(t).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from combine_ep_get_gb300.inputs import CONFIGS, make_config, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_layout(topk_idx, E, R, rpn=0, align=1):
    T, K = topk_idx.shape
    el = E // R
    valid = (topk_idx >= 0) & (topk_idx < E)
    cnt_e = np.bincount(topk_idx[valid], minlength=E).astype(np.int64)
    member = np.zeros((T, R), bool)
    for r in range(R):
        lo, hi = r * el, (r + 1) * el
        member[:, r] = (valid & (topk_idx >= lo) & (topk_idx < hi)).any(axis=1)
    lists = [np.sort(np.flatnonzero(member[:, r])) for r in range(R)]
    pairs = [(r, int(t)) for r in range(R) for t in lists[r]]
    dst = -np.ones((T, R), np.int64)
    for row, (r, t) in enumerate(pairs):
        dst[t, r] = row
    starts = [0]
    for r in range(R):
        starts.append(starts[-1] + len(lists[r]))
    padded = -(-cnt_e // align) * align
    exp_off = np.concatenate([[0], np.cumsum(padded)])
    nodes = None
    if rpn:
        nodes = np.array([member[:, n * rpn:(n + 1) * rpn].any(axis=1).sum() for n in range(R // rpn)])
    src_dst = None
    if T % R == 0:
        ts = T // R
        src_dst = np.array([member[s * ts:(s + 1) * ts].sum(axis=0) for s in range(R)]).reshape(R, R)
    # rows numbered token by token: how many receive lists name each token
    per_tok = np.bincount(np.concatenate(lists + [np.zeros(0, np.int64)]).astype(np.int64), minlength=T)
    tok_off = np.concatenate([[0], np.cumsum(per_tok)])
    return dict(num_tokens_per_expert=cnt_e, num_tokens_per_rank=np.array([len(l) for l in lists]),
                token_offset=tok_off,
                rank_offset=np.array(starts), dst_row=dst, is_token_in_rank=member.astype(np.uint8),
                expert_offset=exp_off, num_tokens_per_node=nodes, src_dst_count=src_dst,
                invalid=bool(((topk_idx < -1) | (topk_idx >= E)).any()))


def check_against(L, ref):
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "dst_row",
                "is_token_in_rank", "expert_offset", "token_offset"):
        np.testing.assert_array_equal(getattr(L, key), ref[key], err_msg=key)
    if ref["num_tokens_per_node"] is not None:
        np.testing.assert_array_equal(L.num_tokens_per_node, ref["num_tokens_per_node"])
    if ref["src_dst_count"] is not None:
        np.testing.assert_array_equal(L.src_dst_count, ref["src_dst_count"])
    assert bool(L.status & oracle.EP_ERR_INVALID_INDEX) == ref["invalid"]


def test_handworked_example():
    g = json.load(open(os.path.join(GOLDEN, "layout_handworked.json")))
    idx = np.array(g["topk_idx"], np.int64)
    L = oracle.layout(idx, g["E"], g["R"], g["ranks_per_node"], g["expert_alignment"])
    assert L.status == 0
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "num_tokens_per_node", "rank_offset",
                "expert_offset", "is_token_in_rank", "dst_row", "src_dst_count", "token_offset"):
        np.testing.assert_array_equal(getattr(L, key), np.array(g[key]), err_msg=key)


@pytest.mark.parametrize("T,K,E,R,rpn,align,mode", [
    (1, 1, 1, 1, 0, 1, "uniform"),
    (7, 3, 12, 3, 0, 1, "uniform"),
    (64, 4, 16, 4, 2, 4, "uniform"),
    (300, 8, 64, 8, 4, 16, "masked"),
    (257, 6, 48, 16, 8, 1, "replace"),     # duplicates and masked entries
    (96, 5, 40, 8, 0, 3, "invalid"),       # out-of-range ids are flagged and skipped
    (33, 2, 32, 32, 4, 1, "uniform"),      # one expert per rank
    (128, 9, 2048, 1024, 0, 1, "uniform"),  # the largest rank count
])
def test_brute_force_small(T, K, E, R, rpn, align, mode):
    rng = np.random.Generator(np.random.PCG64(1000 + T + K + E + R))
    if mode in ("uniform", "masked"):
        idx = make_inputs(T, 8, E, K, R, seed=T * 7 + K, mask_frac=0.2 if mode == "masked" else 0.0,
                          with_x=False)["topk_idx"]
    elif mode == "replace":
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int64)
    else:
        idx = rng.integers(-3, E + 3, size=(T, K)).astype(np.int64)
    L = oracle.layout(idx, E, R, rpn, align)
    check_against(L, brute_layout(idx, E, R, rpn, align))


def test_empty_tokens():
    idx = np.zeros((0, 8), np.int64)
    L = oracle.layout(idx, 256, 8)
    assert L.status == 0
    assert L.num_tokens_per_rank.sum() == 0 and L.rank_offset.tolist() == [0] * 9
    assert L.expert_offset.tolist() == [0] * 257


def test_all_masked_token_and_empty_rank():
    idx = np.array([[-1, -1, -1], [0, 1, 2], [-1, -1, -1], [5, 4, 3]], np.int64)
    L = oracle.layout(idx, 12, 4)          # 3 experts per rank; ranks 2 and 3 get nothing
    np.testing.assert_array_equal(L.num_tokens_per_rank, [1, 1, 0, 0])
    np.testing.assert_array_equal(L.dst_row[0], [-1, -1, -1, -1])
    np.testing.assert_array_equal(L.dst_row[2], [-1, -1, -1, -1])
    np.testing.assert_array_equal(L.dst_row[1], [0, -1, -1, -1])
    np.testing.assert_array_equal(L.dst_row[3], [-1, 1, -1, -1])


def _invariants(L, idx, E, R, rpn):
    T, K = idx.shape
    masked = int((idx == -1).sum())
    assert L.num_tokens_per_expert.sum() == T * K - masked
    n_t = L.is_token_in_rank.sum(axis=1)
    assert L.num_tokens_per_rank.sum() == L.rank_offset[-1] == n_t.sum()
    assert (np.diff(L.rank_offset) == L.num_tokens_per_rank).all()
    assert (np.diff(L.token_offset) == n_t).all() and L.token_offset[-1] == L.rank_offset[-1]
    # each (t, r) in the rank has exactly one row; rows within a rank rise with t
    for r in range(R):
        rows = L.dst_row[:, r]
        ts = np.flatnonzero(L.is_token_in_rank[:, r])
        assert (rows[L.is_token_in_rank[:, r] == 0] == -1).all()
        np.testing.assert_array_equal(rows[ts], L.rank_offset[r] + np.arange(len(ts)))
    if L.src_dst_count is not None:
        np.testing.assert_array_equal(L.src_dst_count.sum(axis=0), L.num_tokens_per_rank)
    if rpn:
        per = L.num_tokens_per_rank.reshape(-1, rpn)
        assert (L.num_tokens_per_node <= per.sum(axis=1)).all()
        assert (L.num_tokens_per_node >= per.max(axis=1)).all()
    return n_t


@pytest.mark.parametrize("name", list(CONFIGS))
def test_invariants_on_workloads(name):
    d = make_config(name, with_x=False)
    c = d["cfg"]
    L = oracle.layout(d["topk_idx"], c.E, c.R, c.ranks_per_node, 1)
    assert L.status == 0
    n_t = _invariants(L, d["topk_idx"], c.E, c.R, c.ranks_per_node)
    if name == "skewed":
        assert int((d["topk_idx"] == -1).sum()) == int(0.05 * c.T * c.K)
    if name == "large":
        nodes_per_token = np.array([len(set((row[row >= 0] // (c.E // (c.R // c.ranks_per_node))).tolist()))
                                    for row in d["topk_idx"][:2000]])
        assert nodes_per_token.max() <= c.max_nodes
    assert n_t.max() <= min(c.K, c.R)


def expected_distinct_groups(E, K, G):
    return G * (1 - math.comb(E - E // G, K) / math.comb(E, K))


@pytest.mark.parametrize("E,K,R,T", [(16, 4, 4, 20000), (256, 8, 8, 20000), (256, 8, 32, 20000),
                                     (256, 8, 64, 20000)])
def test_mean_ranks_per_token_closed_form(E, K, R, T):
    idx = make_inputs(T, 8, E, K, R, seed=E + K + R, with_x=False)["topk_idx"]
    L = oracle.layout(idx, E, R)
    n_t = L.is_token_in_rank.sum(axis=1).astype(np.float64)
    mu = expected_distinct_groups(E, K, R)
    se = n_t.std() / math.sqrt(T)
    assert abs(n_t.mean() - mu) <= 4 * se + 1e-12, (n_t.mean(), mu, se)


def test_node_limited_closed_form():
    # Experts uniform over the 4 chosen nodes' 128 experts = 32 ranks of 4
    # experts each: the expected distinct ranks are 32 (1 - C(124,8)/C(128,8)).
    c = CONFIGS["large"]
    d = make_config("large", with_x=False)
    L = oracle.layout(d["topk_idx"], c.E, c.R, c.ranks_per_node)
    n_t = L.is_token_in_rank.sum(axis=1).astype(np.float64)
    mu = expected_distinct_groups(128, 8, 32)
    assert abs(n_t.mean() - mu) <= 4 * n_t.std() / math.sqrt(c.T)
    nn = L.num_tokens_per_node
    # every token touches between 1 and 4 nodes
    assert c.T <= nn.sum() <= 4 * c.T
