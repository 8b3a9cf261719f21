"""Pins for the CPU oracle's FP8 E4M3 cast (no GPU).

The encoder follows the OCP 8-bit floating point definition (E4M3: bias 7,
3 mantissa bits, subnormals, S.1111.111 = NaN, no infinities, max 448) with
round-to-nearest-even and saturation.  It is pinned by:

* torch's float8_e4m3fn decode of all 256 codes (a library routine);
* round trip of every finite code;
* ties at every midpoint between neighbouring codes go to the even code;
* torch's float32 -> float8_e4m3fn cast on random in-range values;
* the per-128-channel row cast against a torch formulation of
  amax -> sf = amax/448 -> q = e4m3(x * (448/amax)), plus error bounds.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import make_rows


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy()


def test_decode_table_matches_library():
    ours = oracle.e4m3_decode(np.arange(256))
    ref = torch_decode_all()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and (np.flatnonzero(nan) == [0x7F, 0xFF]).all()
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert ref[0x7E] == 448.0 and ref[0x01] == 2.0 ** -9 and ref[0x08] == 2.0 ** -6


def test_round_trip_all_finite_codes():
    ref = torch_decode_all()
    for c in range(256):
        if np.isnan(ref[c]):
            continue
        assert oracle.e4m3_encode([ref[c]])[0] == c, hex(c)


def test_midpoints_round_to_even():
    ref = torch_decode_all()
    pos = [(ref[c], c) for c in range(0x7F)]            # +0 .. 448, ascending
    for (a, ca), (b, cb) in zip(pos[:-1], pos[1:]):
        mid = np.float32((np.float64(a) + np.float64(b)) / 2)
        assert float(mid) == (float(a) + float(b)) / 2     # midpoints are exact in fp32
        want = ca if ca % 2 == 0 else cb
        assert oracle.e4m3_encode([mid])[0] == want
        assert oracle.e4m3_encode([-mid])[0] == (want | 0x80)


def test_saturation_and_nan():
    enc = oracle.e4m3_encode([448.0, 464.0, 1e6, 3.4e38, -500.0, np.nan])
    assert enc.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F]


def test_against_library_cast_random():
    rng = np.random.Generator(np.random.PCG64(123))
    v = np.concatenate([
        rng.uniform(-447.0, 447.0, 4000),
        rng.standard_normal(4000) * 0.01,
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 4000),        # subnormal range
    ]).astype(np.float32)
    ours = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_row_cast_against_torch_formulation():
    H = 7168
    x = make_rows(4, H, seed=21)
    x[1, :128] = 0                                        # an all-zero block
    x[2, 128:256] = 0x8000                                # negative zeros
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    for i in range(4):
        q, sf = oracle.fp8_cast_row(x[i])
        blocks = xf[i].view(-1, 128)
        amax = blocks.abs().amax(dim=1)
        safe = torch.where(amax > 0, amax, torch.ones_like(amax))
        c448 = torch.full_like(safe, 448.0)
        # tensor / tensor is an IEEE divide; ``448.0 / tensor`` is not (torch
        # evaluates it as reciprocal(tensor) * 448, two roundings)
        sf_ref = torch.where(amax > 0, safe / c448, torch.ones_like(amax))
        mult = torch.where(amax > 0, c448 / safe, torch.zeros_like(amax))
        q_ref = (blocks * mult[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(-1).numpy()
        np.testing.assert_array_equal(sf, sf_ref.numpy())
        np.testing.assert_array_equal(q, q_ref)
        # error bounds: normal-range codes within 2^-4 relative; subnormal codes
        # within half the subnormal step 2^-10 (times the block scale)
        deq = oracle.e4m3_decode(q).reshape(-1, 128).astype(np.float64) * sf.astype(np.float64)[:, None]
        xb = blocks.numpy().astype(np.float64)
        scaled = np.abs(xb) * (448.0 / np.where(amax.numpy() > 0, amax.numpy(), 1.0))[:, None]
        normal = scaled >= 2.0 ** -6
        err = np.abs(deq - xb)
        assert (err[normal] <= 2.0 ** -4 * np.abs(xb[normal]) * 1.0001).all()
        bound = (2.0 ** -10 * sf.astype(np.float64))[:, None] * np.ones_like(xb)
        assert (err[~normal] <= bound[~normal] * 1.0001).all()
    q, sf = oracle.fp8_cast_row(x[1])
    assert sf[0] == 1.0 and (q[:128] == 0).all()
    q, sf = oracle.fp8_cast_row(x[2])
    assert sf[1] == 1.0 and (q[128:256] == 0x80).all()
