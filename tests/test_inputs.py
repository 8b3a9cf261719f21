"""The seeded input generator: determinism and the workload shapes (no GPU)."""
import numpy as np

from combine_ep_get_gb300.inputs import CONFIGS, make_config, make_inputs, make_rows


def test_deterministic_and_x_independent():
    a = make_inputs(64, 256, 16, 4, 4, seed=9)
    b = make_inputs(64, 256, 16, 4, 4, seed=9)
    c = make_inputs(64, 256, 16, 4, 4, seed=9, with_x=False)
    for k in ("topk_idx", "topk_weights", "x_bits"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(a["topk_idx"], c["topk_idx"])
    assert a["x_bits"].dtype == np.uint16 and a["topk_idx"].dtype == np.int64


def test_distinct_experts_and_weights():
    for name in ("tiny", "dsv3", "decode", "large"):
        d = make_config(name, with_x=False)
        c = d["cfg"]
        idx = d["topk_idx"]
        assert idx.shape == (c.T, c.K) and idx.min() >= 0 and idx.max() < c.E
        s = np.sort(idx, axis=1)
        assert (np.diff(s, axis=1) > 0).all()
        np.testing.assert_allclose(d["topk_weights"].sum(axis=1), 1.0, rtol=1e-5)


def test_skewed_routing_shape():
    d = make_config("skewed", with_x=False)
    c = d["cfg"]
    idx = d["topk_idx"]
    assert int((idx == -1).sum()) == int(np.floor(0.05 * c.T * c.K)) == 3276
    counts = np.bincount(idx[idx >= 0], minlength=c.E)
    # Zipf(1.2): the hottest expert takes far more than the uniform share
    assert counts.max() > 10 * (c.T * c.K / c.E)
    for row in idx[:500]:
        v = row[row >= 0]
        assert len(set(v.tolist())) == len(v)


def test_rows_bf16():
    y = make_rows(3, 128, seed=1)
    assert y.shape == (3, 128) and y.dtype == np.uint16
    f = (y.astype(np.uint32) << 16).view(np.float32)
    assert np.isfinite(f).all() and 0.5 < f.std() < 1.5


def test_configs_cover_workloads():
    assert set(CONFIGS) == {"tiny", "dsv3", "skewed", "decode", "large"}
    assert CONFIGS["decode"].fp8 and CONFIGS["decode"].weighted
    assert CONFIGS["large"].ranks_per_node == 8
