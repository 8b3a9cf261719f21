"""GPU parity of the routing layout against the CPU oracle: bit-exact on all
five workloads at full size, plus ragged, masked, invalid and limit cases."""
import numpy as np
import pytest

import oracle
from combine_ep_get_gb300.inputs import CONFIGS, make_config, make_inputs

pytestmark = pytest.mark.gpu

FIELDS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_offset",
          "expert_offset", "dst_row", "token_offset")


def _compare(idx, E, R, rpn=0, align=1):
    from gpu_path import layout_host, run_layout
    lay, status = run_layout(idx, E, R, rpn, align)
    g = layout_host(lay)
    o = oracle.layout(idx, E, R, rpn, align)
    for f in FIELDS:
        np.testing.assert_array_equal(g[f], getattr(o, f), err_msg=f)
    if rpn:
        np.testing.assert_array_equal(g["num_tokens_per_node"], o.num_tokens_per_node)
    if o.src_dst_count is not None:
        np.testing.assert_array_equal(g["src_dst_count"], o.src_dst_count)
    assert int(status.item()) == o.status
    return g, o


@pytest.mark.parametrize("name", list(CONFIGS))
def test_layout_workloads_full_size(name):
    d = make_config(name, with_x=False)
    c = d["cfg"]
    _compare(d["topk_idx"], c.E, c.R, c.ranks_per_node, 1)


@pytest.mark.parametrize("T,K,E,R,rpn,align,mask", [
    (1, 8, 256, 8, 0, 1, 0.0),
    (255, 8, 256, 8, 2, 1, 0.0),
    (257, 8, 256, 16, 4, 128, 0.05),
    (1000, 6, 96, 12, 3, 7, 0.3),
    (4096 + 77, 8, 256, 64, 8, 1, 0.02),
    (64, 4, 64, 64, 0, 1, 0.0),           # one expert per rank
    (300, 3, 32, 1, 0, 1, 0.0),           # one rank
    (512, 32, 2048, 1024, 32, 1, 0.0),    # the limits: R=1024, E=2048, K=32
    (2048, 9, 2048, 8, 0, 16, 0.1),       # 256 experts per rank
    (4096, 8, 2048, 1024, 0, 1, 0.0),     # many (token, rank) outputs: tiled path
    (32768, 8, 256, 128, 16, 1, 0.01),    # tiled path with node and source counts
    (9000, 8, 256, 256, 32, 3, 0.0),      # tiled path, ragged last tile
    # single-CTA path (T <= 1024, R <= 32, K <= 16) at and around its limits
    (1024, 16, 512, 32, 8, 1, 0.1),       # 32 words x 32 ranks, K = 16
    (1025, 8, 256, 32, 0, 1, 0.0),        # one token over: cluster path
    (1000, 17, 256, 8, 0, 1, 0.0),        # K = 17: cluster path
    (200, 5, 30, 3, 0, 1, 0.1),           # R = 3: byte-wise rows of is_token_in_rank
    (96, 8, 256, 32, 32, 1, 0.0),         # one node; source ranks of 3 tokens cross words
    (33, 8, 64, 32, 1, 2, 0.0),           # 32 nodes of one rank, ragged second word
    (500, 8, 2048, 32, 4, 5, 0.05),       # 64 expert chunks, alignment 5
])
def test_layout_shapes(T, K, E, R, rpn, align, mask):
    idx = make_inputs(T, 8, E, K, R, seed=T + K + E + R, mask_frac=mask, with_x=False)["topk_idx"]
    _compare(idx, E, R, rpn, align)


def test_layout_duplicates_all_masked_and_invalid():
    rng = np.random.Generator(np.random.PCG64(5))
    idx = rng.integers(-1, 64, size=(777, 8)).astype(np.int64)   # duplicates allowed
    idx[10] = -1                                                  # fully masked token
    idx[20, 3] = 64                                               # invalid
    idx[21, 0] = -5                                               # invalid
    g, o = _compare(idx, 64, 8, 2, 1)
    assert o.status == oracle.EP_ERR_INVALID_INDEX
    assert (g["dst_row"][10] == -1).all()


def test_layout_empty():
    idx = np.zeros((0, 8), np.int64)
    g, o = _compare(idx, 256, 8, 0, 1)
    assert g["rank_offset"].tolist() == [0] * 9


def test_layout_rank_without_tokens():
    idx = make_inputs(500, 8, 64, 4, 8, seed=3, with_x=False)["topk_idx"]
    idx = np.where((idx >= 16) & (idx < 24), -1, idx)                # rank 2 gets nothing
    g, o = _compare(idx, 64, 8, 4, 1)
    assert g["num_tokens_per_rank"][2] == 0
