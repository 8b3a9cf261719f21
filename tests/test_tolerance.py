"""The combine tolerance separates fp32 from bf16 accumulation (no GPU).

On the decode workload (T=128, H=7168, E=256, K=8, R=32, weighted) and on a
1000 x 7168 weighted shape (E=256, K=8, R=8), two numpy emulations of the
combine are compared with the oracle's exact sum:
- fp32 accumulation (coefficients summed in fp32, one fp32 rounding per
  accumulated product, one bf16 rounding at the end) must pass both bounds
  everywhere;
- an accumulator kept in bf16 (a bf16 rounding after every accumulated
  product) must break the fp32-accumulation bound, while it mostly passes the
  1e-2 bound -- which is why both are checked.
"""
import numpy as np
import pytest

import oracle
from combine_ep_get_gb300.inputs import make_config, make_inputs, make_rows
from tolerance import bf16_bits_to_f64, check_close, combine_bounds, rank_sources


def _emulate(y_bits, idx, w, E, R, dst_row, acc_bf16):
    """Combine in ascending rank order with an fp32 or a bf16 accumulator."""
    T, K = idx.shape
    H = y_bits.shape[1]
    el = E // R
    acc = np.zeros((T, H), np.float64)
    for r in range(R):
        d = dst_row[:, r]
        ok = d >= 0
        if not ok.any():
            continue
        c = np.zeros(T, np.float32)
        for k in range(K):
            on = ok & (idx[:, k] >= 0) & (idx[:, k] // el == r)
            c = np.where(on, (c + w[:, k]).astype(np.float32), c)
        prod = c.astype(np.float64)[ok, None] * bf16_bits_to_f64(y_bits[d[ok]])   # exact in fp64
        s = acc[ok] + prod
        if acc_bf16:
            acc[ok] = bf16_bits_to_f64(oracle.double_to_bf16(s.ravel()).reshape(s.shape))
        else:
            acc[ok] = s.astype(np.float32).astype(np.float64)
    if acc_bf16:
        return oracle.double_to_bf16(acc.ravel()).reshape(T, H)
    return oracle.float_to_bf16(acc.astype(np.float32).ravel()).reshape(T, H)


def _case(name):
    if name == "decode":
        d = make_config("decode", with_x=False)
        c = d["cfg"]
        return d["topk_idx"], d["topk_weights"], c.E, c.R, c.H, 3
    T, H, E, K, R = 1000, 7168, 256, 8, 8
    d = make_inputs(T, H, E, K, R, seed=T + 5 * H, with_x=False)
    return d["topk_idx"], d["topk_weights"], E, R, H, 4


@pytest.mark.parametrize("name", ["decode", "1000x7168"])
def test_bound_separates_fp32_from_bf16_accumulation(name):
    idx, w, E, R, H, seed = _case(name)
    L = oracle.layout(idx, E, R)
    y_bits = make_rows(L.num_recv, H, seed=seed)
    ref, st = oracle.combine(y_bits, idx, w, E, R, L.dst_row, weighted=True)
    assert st == 0
    rows, c, a, m = rank_sources(idx, w, E, R, L.dst_row, True)
    loose, tight = combine_bounds(y_bits, rows, c, a, ref, m)

    fp32 = _emulate(y_bits, idx, w, E, R, L.dst_row, acc_bf16=False)
    check_close(fp32, ref, loose, tight)

    bf16 = _emulate(y_bits, idx, w, E, R, L.dst_row, acc_bf16=True)
    err = np.abs(bf16_bits_to_f64(bf16) - ref)
    frac_tight = float((err > tight).mean())
    frac_loose = float((err > loose).mean())
    assert frac_tight > 0.05, frac_tight       # the tight bound rejects bf16 accumulation
    assert frac_loose < 0.01, frac_loose       # the 1e-2 bound alone would not


def test_bound_is_not_loose_by_orders_of_magnitude():
    """The fp32 emulation's error comes within 2^-2 of the bound somewhere:
    the bound is the bf16 rounding itself, not a large multiple of it."""
    idx, w, E, R, H, seed = _case("decode")
    L = oracle.layout(idx, E, R)
    y_bits = make_rows(L.num_recv, H, seed=seed)
    ref, _ = oracle.combine(y_bits, idx, w, E, R, L.dst_row, weighted=True)
    rows, c, a, m = rank_sources(idx, w, E, R, L.dst_row, True)
    _, tight = combine_bounds(y_bits, rows, c, a, ref, m)
    fp32 = _emulate(y_bits, idx, w, E, R, L.dst_row, acc_bf16=False)
    ratio = np.abs(bf16_bits_to_f64(fp32) - ref) / tight
    assert ratio.max() > 0.25
