"""GPU parity of combine against the CPU oracle.

Tolerance (fp32 accumulation, bf16 output), elementwise against the oracle's
fp64 sum: |gpu - oracle| <= 1e-2 * sum_r |c(t,r) * y_r|, and the tighter bound
of fp32 accumulation with one bf16 rounding (tests/tolerance.py).
The unweighted identity round trip has a closed form that must hold exactly
(as values) in any summation order: out[t] = bf16(n(t) * x[t]).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import CONFIGS, make_config, make_inputs, make_rows
from tolerance import check_close, rank_combine_bounds

pytestmark = pytest.mark.gpu


def _setup(d, E, R, rpn=0):
    from gpu_path import run_layout, to_dev
    idx = to_dev(d["topk_idx"])
    w = to_dev(d["topk_weights"])
    lay, st = run_layout(idx, E, R, rpn)
    return idx, w, lay


@pytest.mark.parametrize("T,H,E,K,R,mask,weighted", [
    (128, 256, 16, 4, 4, 0.0, False),
    (1000, 7168, 256, 8, 8, 0.0, False),
    (1000, 7168, 256, 8, 8, 0.0, True),
    (777, 2048, 64, 6, 16, 0.2, True),
    (300, 8, 32, 2, 32, 0.0, False),
    (33, 4096, 128, 8, 64, 0.05, True),
    (300, 512, 256, 8, 128, 0.0, True),      # more than 64 ranks
    (200, 256, 2048, 32, 1024, 0.1, True),   # the limits: 1024 ranks, top-32
])
def test_combine_random_rows(T, H, E, K, R, mask, weighted):
    from gpu_path import bf16_bits, run_combine, x_tensor
    d = make_inputs(T, H, E, K, R, seed=T + 5 * H, mask_frac=mask, with_x=False)
    idx, w, lay = _setup(d, E, R)
    n = lay.num_recv
    y_bits = make_rows(n, H, seed=T + H + 1)
    out, st = run_combine(x_tensor(y_bits), idx, w if weighted else None, E, R, lay, T, H)
    assert int(st.item()) == 0
    L = oracle.layout(d["topk_idx"], E, R)
    ref, _ = oracle.combine(y_bits, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, weighted=weighted)
    loose, tight = rank_combine_bounds(y_bits, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, weighted, ref)
    check_close(bf16_bits(out), ref, loose, tight)
    # tokens that reach no rank come back as zero rows
    none = L.is_token_in_rank.sum(axis=1) == 0
    assert (bf16_bits(out)[none] == 0).all()


@pytest.mark.parametrize("name", ["tiny", "dsv3", "skewed", "large"])
def test_round_trip_identity_closed_form(name):
    """dispatch -> identity expert -> combine == bf16(n(t) * x[t]), bit-exact, all tokens."""
    from gpu_path import run_combine, run_dispatch, to_dev, x_tensor
    d = make_config(name)
    c = d["cfg"]
    idx, w, lay = _setup(d, c.E, c.R, c.ranks_per_node)
    x = x_tensor(d["x_bits"])
    n = lay.num_recv
    res = run_dispatch(x, idx, w, c.E, c.R, lay, n)
    out, st = run_combine(res["recv_x"], idx, None, c.E, c.R, lay, c.T, c.H)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(res["status"].item()) == 0
    nt = lay.is_token_in_rank.sum(dim=1, dtype=torch.int32).float()
    want = (x.float() * nt[:, None]).to(torch.bfloat16)
    # exact values (bf16 -> fp32 is exact); a sum of -0 terms started from +0 is
    # +0 while n * (-0) is -0, so compare values, not sign bits of zeros
    assert torch.equal(out.float(), want.float())


@pytest.mark.parametrize("name", ["dsv3", "skewed", "large"])
def test_combine_full_size_sampled(name):
    from gpu_path import bf16_bits, run_combine, x_tensor
    d = make_config(name, with_x=False)
    c = d["cfg"]
    idx, w, lay = _setup(d, c.E, c.R, c.ranks_per_node)
    n = lay.num_recv
    y_bits = make_rows(n, c.H, seed=c.seed + 100)
    out, st = run_combine(x_tensor(y_bits), idx, None, c.E, c.R, lay, c.T, c.H)
    assert int(st.item()) == 0
    L = oracle.layout(d["topk_idx"], c.E, c.R)
    rng = np.random.Generator(np.random.PCG64(7))
    toks = np.unique(np.concatenate([[0, c.T - 1], rng.choice(c.T, 40, replace=False)])).astype(np.int32)
    ref, _ = oracle.combine(y_bits, d["topk_idx"], None, c.E, c.R, L.dst_row, tokens=toks)
    loose, tight = rank_combine_bounds(y_bits, d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row, False, ref,
                                       tokens=toks)
    check_close(bf16_bits(out)[toks], ref, loose, tight)


def test_decode_fp8_weighted_round_trip():
    """Decode workload: FP8 dispatch, identity expert on the dequantised rows,
    weighted combine, against the oracle run on the oracle's own dispatch."""
    from gpu_path import run_combine, run_dispatch, x_tensor, bf16_bits
    d = make_config("decode")
    c = d["cfg"]
    idx, w, lay = _setup(d, c.E, c.R)
    x = x_tensor(d["x_bits"])
    n = lay.num_recv
    res = run_dispatch(x, idx, w, c.E, c.R, lay, n, fp8=True)
    # identity expert: dequantise codes * per-block scale, rounded to bf16 (test harness)
    q = res["recv_x"][:n].view(torch.float8_e4m3fn).float()
    sf = res["recv_sf"][:n * (c.H // 128)].view(n, -1)
    y = (q.view(n, -1, 128) * sf[:, :, None]).view(n, c.H).to(torch.bfloat16).contiguous()
    out, st = run_combine(y, idx, w, c.E, c.R, lay, c.T, c.H)
    assert int(st.item()) == 0
    L = oracle.layout(d["topk_idx"], c.E, c.R)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row, fp8=True)
    deq = oracle.e4m3_decode(o["recv_x"].ravel()).reshape(n, -1, 128).astype(np.float64)
    y_ref = (deq * o["recv_sf"].astype(np.float64)[:, :, None]).reshape(n, c.H).astype(np.float32)
    y_ref_bits = oracle.float_to_bf16(y_ref).reshape(n, c.H)
    ref, _ = oracle.combine(y_ref_bits, d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row, weighted=True)
    loose, tight = rank_combine_bounds(y_ref_bits, d["topk_idx"], d["topk_weights"], c.E, c.R, L.dst_row, True,
                                       ref)
    check_close(bf16_bits(out), ref, loose, tight)


def test_combine_capacity_flag():
    from gpu_path import run_combine, x_tensor
    T, H, E, K, R = 200, 256, 32, 4, 8
    d = make_inputs(T, H, E, K, R, seed=4, with_x=False)
    idx, w, lay = _setup(d, E, R)
    n = lay.num_recv
    y_bits = make_rows(n - 10, H, seed=2)
    out, st = run_combine(x_tensor(y_bits), idx, None, E, R, lay, T, H)
    assert int(st.item()) & oracle.EP_ERR_CAPACITY
    L = oracle.layout(d["topk_idx"], E, R)
    ref, _ = oracle.combine(y_bits, d["topk_idx"], None, E, R, L.dst_row)
    from gpu_path import bf16_bits
    # rows beyond the capacity are skipped on both sides
    loose, tight = rank_combine_bounds(y_bits, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, False, ref,
                                       num_y_rows=n - 10)
    check_close(bf16_bits(out), ref, loose, tight)


@pytest.mark.parametrize("T,E,K,R,mask", [(4096, 256, 8, 8, 0.0), (777, 64, 6, 16, 0.2), (200, 2048, 32, 1024, 0.1)])
def test_combined_topk_weights(T, E, K, R, mask):
    """Bit-exact against the oracle (same fp32 order); for unmodified received
    weights, exactly topk_weights on valid slots and 0 on masked ones."""
    from gpu_path import B, run_dispatch, to_dev, x_tensor
    d = make_inputs(T, 16, E, K, R, seed=T + E, mask_frac=mask)
    idx, w, lay = _setup(d, E, R)
    n = lay.num_recv
    res = run_dispatch(x_tensor(d["x_bits"]), idx, w, E, R, lay, n)
    rw = res["recv_topk_weights"]
    rw_mod = (rw * 0.75 + 0.125).contiguous()          # weights an expert might rewrite
    L = oracle.layout(d["topk_idx"], E, R)
    for src, scale in ((rw, None), (rw_mod, True)):
        comb = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.ep_combine_topk_weights(src, E, R, lay, comb, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref, _ = oracle.combine_topk_weights(src.cpu().numpy(), L.dst_row)
        np.testing.assert_array_equal(comb.cpu().numpy(), ref)
        if scale is None:
            want = np.where(d["topk_idx"] >= 0, d["topk_weights"], 0.0).astype(np.float32)
            np.testing.assert_array_equal(comb.cpu().numpy(), want)


def test_expert_stats_accumulate():
    from gpu_path import B
    d = make_config("skewed", with_x=False)
    c = d["cfg"]
    idx, w, lay = _setup(d, c.E, c.R)
    stats = torch.zeros(c.E, dtype=torch.int64, device="cuda")
    B.ep_accumulate_expert_stats(lay, c.E, stats)
    B.ep_accumulate_expert_stats(lay, c.E, stats)
    torch.cuda.synchronize()
    L = oracle.layout(d["topk_idx"], c.E, c.R)
    ref = np.zeros(c.E, np.int64)
    oracle.accumulate_expert_stats(L.num_tokens_per_expert, ref)
    oracle.accumulate_expert_stats(L.num_tokens_per_expert, ref)
    np.testing.assert_array_equal(stats.cpu().numpy(), ref)
