"""GPU parity of dispatch against the CPU oracle.

* element by element (payload bytes, scales, remapped top-k, weights, source
  index) at sizes the oracle finishes in seconds, spanning several tiles and a
  ragged tail;
* at the full workload sizes, in the bench's launch configuration: the
  metadata of every row against the oracle run on a 16-channel stand-in row
  (metadata does not depend on the payload), the payload of sampled tokens
  against the oracle's sampled dispatch, and recv_x[d] == x[src[d]] for every
  row;
* FP8 (decode workload, full size): codes and scales bit-exact;
* capacity overflow and invalid ids set the status and leave other rows right.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import CONFIGS, make_config, make_inputs

pytestmark = pytest.mark.gpu


def _run(d, E, R, fp8=False, sf_col_major=False, capacity=None, rpn=0):
    from gpu_path import run_dispatch, run_layout, to_dev, x_tensor
    idx = to_dev(d["topk_idx"])
    w = to_dev(d["topk_weights"])
    x = x_tensor(d["x_bits"])
    lay, st = run_layout(idx, E, R, rpn)
    n = lay.num_recv
    cap = n if capacity is None else capacity
    res = run_dispatch(x, idx, w, E, R, lay, cap, fp8=fp8, sf_col_major=sf_col_major)
    torch.cuda.synchronize()
    return lay, res, n, x, idx


def _host(res, fp8, n):
    from gpu_path import bf16_bits
    out = dict(recv_topk_idx=res["recv_topk_idx"][:n].cpu().numpy(),
               recv_topk_weights=res["recv_topk_weights"][:n].cpu().numpy(),
               recv_src_idx=res["recv_src_idx"][:n].cpu().numpy())
    if fp8:
        out["recv_x"] = res["recv_x"][:n].cpu().numpy()
    else:
        out["recv_x"] = bf16_bits(res["recv_x"][:n]).view(np.uint8).reshape(n, -1)
    return out


@pytest.mark.parametrize("T,H,E,K,R,mask", [
    (128, 256, 16, 4, 4, 0.0),        # the small workload's shape
    (1000, 7168, 256, 8, 8, 0.0),     # 4 tiles, ragged tail, DeepSeek-V3 row
    (777, 2048, 64, 6, 16, 0.1),
    (300, 8, 32, 2, 32, 0.0),         # 16-byte rows
    (33, 4096, 128, 8, 64, 0.05),     # few tokens: rows split into pieces
    (1, 7168, 256, 8, 8, 0.0),
    (300, 512, 256, 8, 128, 0.0),     # more than 64 ranks
    (200, 256, 2048, 32, 1024, 0.1),  # the limits: 1024 ranks, top-32
])
def test_dispatch_bf16_full_compare(T, H, E, K, R, mask):
    d = make_inputs(T, H, E, K, R, seed=T * 3 + H, mask_frac=mask)
    lay, res, n, _, _ = _run(d, E, R)
    assert int(res["status"].item()) == 0
    g = _host(res, False, n)
    L = oracle.layout(d["topk_idx"], E, R)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row)
    for k in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)


@pytest.mark.parametrize("name", ["dsv3", "skewed", "large"])
def test_dispatch_bf16_full_size_sampled(name):
    d = make_config(name)
    c = d["cfg"]
    lay, res, n, x, idx = _run(d, c.E, c.R, rpn=c.ranks_per_node)
    assert int(res["status"].item()) == 0
    L = oracle.layout(d["topk_idx"], c.E, c.R)
    assert n == L.num_recv
    # metadata of every row: payload-independent, so the oracle runs on 16-channel rows
    stand_in = np.zeros((c.T, 16), np.uint16)
    om = oracle.dispatch(stand_in, d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row)
    np.testing.assert_array_equal(res["recv_src_idx"][:n].cpu().numpy(), om["recv_src_idx"])
    np.testing.assert_array_equal(res["recv_topk_idx"][:n].cpu().numpy(), om["recv_topk_idx"])
    np.testing.assert_array_equal(res["recv_topk_weights"][:n].cpu().numpy(), om["recv_topk_weights"])
    # every payload row equals its source row (a property at any size)
    src = res["recv_src_idx"][:n].long()
    assert torch.equal(res["recv_x"][:n].view(torch.int16), x.view(torch.int16)[src])
    # sampled tokens against the oracle's own dispatch of those tokens
    rng = np.random.Generator(np.random.PCG64(99))
    toks = np.unique(np.concatenate([[0, c.T - 1], rng.choice(c.T, 48, replace=False)])).astype(np.int32)
    os_ = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row, tokens=toks)
    rows = torch.from_numpy(os_["rows"].astype(np.int64)).cuda()
    from gpu_path import bf16_bits
    got = bf16_bits(res["recv_x"][rows]).view(np.uint8).reshape(len(os_["rows"]), -1)
    np.testing.assert_array_equal(got, os_["recv_x"])


@pytest.mark.parametrize("sf_col_major", [False, True])
def test_dispatch_fp8_decode_full_size(sf_col_major):
    d = make_config("decode")
    c = d["cfg"]
    lay, res, n, _, _ = _run(d, c.E, c.R, fp8=True, sf_col_major=sf_col_major)
    assert int(res["status"].item()) == 0
    g = _host(res, True, n)
    L = oracle.layout(d["topk_idx"], c.E, c.R)
    stride = (n + 3) // 4 * 4
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row, fp8=True,
                        sf_col_major=sf_col_major, sf_stride=stride)
    for k in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)
    sf = res["recv_sf"].cpu().numpy()
    if sf_col_major:
        nb = c.H // 128
        got = sf[:nb * stride].reshape(nb, stride)[:, :n]
        want = o["recv_sf"][:nb * stride].reshape(nb, stride)[:, :n]
    else:
        got = sf[:n * (c.H // 128)].reshape(n, -1)
        want = o["recv_sf"]
    np.testing.assert_array_equal(got, want)


def test_dispatch_fp8_special_blocks():
    T, H, E, K, R = 300, 1024, 64, 8, 8
    d = make_inputs(T, H, E, K, R, seed=8)
    x = d["x_bits"]
    x[0, :128] = 0                     # all-zero block
    x[1, 128:256] = 0x8000             # negative zeros
    x[2, :] = x[2, :] & 0x807F         # tiny values (exponent field 0: subnormal bf16)
    x[2, :] |= 0x0080                  # smallest normal exponent
    x[3, 256:384] = 0x4380             # constant 256.0
    lay, res, n, _, _ = _run(d, E, R, fp8=True)
    g = _host(res, True, n)
    L = oracle.layout(d["topk_idx"], E, R)
    o = oracle.dispatch(x, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, fp8=True)
    np.testing.assert_array_equal(g["recv_x"], o["recv_x"])
    sf = res["recv_sf"].cpu().numpy()[:n * (H // 128)].reshape(n, -1)
    np.testing.assert_array_equal(sf, o["recv_sf"])


def _every_amax_x(T, H, seed):
    """bf16 rows whose 128-channel blocks take, in order, every finite bf16
    magnitude 0x0000..0x7f7f as their amax (at a random channel, random sign);
    the block's other channels are random magnitudes up to it."""
    rng = np.random.default_rng(seed)
    nb = H // 128
    amax = np.arange(0x7F80, dtype=np.int64)
    blocks = np.zeros((T * nb, 128), np.int64)
    n = min(len(amax), T * nb)
    blocks[:n] = (rng.random((n, 128)) * (amax[:n, None] + 1)).astype(np.int64)
    pos = rng.integers(0, 128, n)
    blocks[np.arange(n), pos] = amax[:n]
    blocks |= rng.integers(0, 2, blocks.shape) << 15
    return blocks.reshape(T, H).astype(np.uint16)


@pytest.mark.parametrize("H,many_tokens", [(2048, True), (7168, False)])
def test_dispatch_fp8_every_amax(H, many_tokens):
    """Codes and scales bit-exact for blocks covering every finite bf16 amax,
    in the many-token mode (8 lanes per block) and the few-token mode (16)."""
    nb = H // 128
    T = (0x7F80 + nb - 1) // nb
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (T >= 8 * sms) == many_tokens
    E, K, R = 64, 4, 8
    d = make_inputs(T, H, E, K, R, seed=40 + nb)
    d["x_bits"] = _every_amax_x(T, H, seed=41 + nb)
    lay, res, n, _, _ = _run(d, E, R, fp8=True)
    assert int(res["status"].item()) == 0
    g = _host(res, True, n)
    L = oracle.layout(d["topk_idx"], E, R)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, fp8=True)
    np.testing.assert_array_equal(g["recv_x"], o["recv_x"])
    sf = res["recv_sf"].cpu().numpy()[:n * nb].reshape(n, -1)
    np.testing.assert_array_equal(sf, o["recv_sf"])


def test_dispatch_capacity_overflow():
    T, H, E, K, R = 400, 512, 64, 4, 8
    d = make_inputs(T, H, E, K, R, seed=12)
    L = oracle.layout(d["topk_idx"], E, R)
    cap = L.num_recv - 50
    lay, res, n, _, _ = _run(d, E, R, capacity=cap)
    assert int(res["status"].item()) & oracle.EP_ERR_CAPACITY
    g = _host(res, False, cap)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, capacity=cap)
    for k in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(g[k], o[k][:cap], err_msg=k)


@pytest.mark.parametrize("T,H,E,K,R", [(64, 1024, 256, 8, 128), (200, 512, 2048, 32, 1024), (7, 128, 16, 2, 4)])
def test_dispatch_fp8_shapes(T, H, E, K, R):
    d = make_inputs(T, H, E, K, R, seed=T + R)
    lay, res, n, _, _ = _run(d, E, R, fp8=True)
    assert int(res["status"].item()) == 0
    g = _host(res, True, n)
    L = oracle.layout(d["topk_idx"], E, R)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, fp8=True)
    for k in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)
    sf = res["recv_sf"].cpu().numpy()[:n * (H // 128)].reshape(n, -1)
    np.testing.assert_array_equal(sf, o["recv_sf"])


@pytest.mark.parametrize("sf_col_major", [False, True])
def test_dispatch_fp8_wide_full_size(sf_col_major):
    """FP8 dispatch with many tokens (8 lanes per 128-channel block, the mode
    timed on the DeepSeek-V3-shaped workload): codes and scales of sampled
    tokens against the oracle's compact dispatch, metadata of every row."""
    import dataclasses
    from combine_ep_get_gb300.inputs import CONFIGS
    d = make_config(dataclasses.replace(CONFIGS["dsv3"], fp8=True))
    c = d["cfg"]
    lay, res, n, _, _ = _run(d, c.E, c.R, fp8=True, sf_col_major=sf_col_major)
    assert int(res["status"].item()) == 0
    L = oracle.layout(d["topk_idx"], c.E, c.R)
    stand_in = np.zeros((c.T, 16), np.uint16)
    om = oracle.dispatch(stand_in, d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row)
    np.testing.assert_array_equal(res["recv_src_idx"][:n].cpu().numpy(), om["recv_src_idx"])
    np.testing.assert_array_equal(res["recv_topk_idx"][:n].cpu().numpy(), om["recv_topk_idx"])
    np.testing.assert_array_equal(res["recv_topk_weights"][:n].cpu().numpy(), om["recv_topk_weights"])
    rng = np.random.Generator(np.random.PCG64(7))
    toks = np.unique(np.concatenate([[0, c.T - 1], rng.choice(c.T, 40, replace=False)])).astype(np.int32)
    os_ = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row, fp8=True,
                          tokens=toks)
    rows = os_["rows"].astype(np.int64)
    np.testing.assert_array_equal(res["recv_x"][torch.from_numpy(rows).cuda()].cpu().numpy(), os_["recv_x"])
    nb = c.H // 128
    sf = res["recv_sf"].cpu().numpy()
    if sf_col_major:
        stride = (n + 3) // 4 * 4
        got = sf[:nb * stride].reshape(nb, stride)[:, rows].T
    else:
        got = sf[:n * nb].reshape(n, nb)[rows]
    np.testing.assert_array_equal(got, os_["recv_sf"])


@pytest.mark.parametrize("T,H,E,K,R,mask,sf_col_major", [
    (1300, 9216, 256, 8, 128, 0.05, False),   # two passes of blocks per row; ranks beyond 64
    (2000, 128, 64, 6, 8, 0.0, True),         # one block per row: most consumer warps idle
    (1216, 16384, 64, 4, 64, 0.1, False),     # 32 KB rows: a shorter ring
    (1500, 1024, 32, 32, 32, 0.3, True),      # top-32, masked entries
])
def test_dispatch_fp8_many_token_shapes(T, H, E, K, R, mask, sf_col_major):
    """FP8 dispatch with at least 8 tokens per SM (the persistent ring kernel)
    on shapes beside the timed one: every code, scale and metadata entry
    against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert T >= 8 * sms
    d = make_inputs(T, H, E, K, R, seed=T + H + K, mask_frac=mask)
    lay, res, n, _, _ = _run(d, E, R, fp8=True, sf_col_major=sf_col_major)
    assert int(res["status"].item()) == 0
    g = _host(res, True, n)
    L = oracle.layout(d["topk_idx"], E, R)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, fp8=True,
                        sf_col_major=sf_col_major, sf_stride=(n + 3) // 4 * 4)
    for k in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)
    nb = H // 128
    if sf_col_major:
        stride = (n + 3) // 4 * 4
        np.testing.assert_array_equal(res["recv_sf"].cpu().numpy()[:nb * stride].reshape(nb, stride)[:, :n],
                                      o["recv_sf"][:nb * stride].reshape(nb, stride)[:, :n])
    else:
        np.testing.assert_array_equal(res["recv_sf"].cpu().numpy()[:n * nb].reshape(n, -1), o["recv_sf"])
