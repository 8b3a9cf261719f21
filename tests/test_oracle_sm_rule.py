"""Pins for the oracle's SM count rule (the ``get_theoretical_num_sms``
fragment of "DeepEP V2 ElasticBuffer architecture", with its
``get_expected_topk`` helper):

* the expected number of distinct ranks per token against brute force over
  every K-subset of experts on tiny shapes (exact rationals), and its closed
  forms K = 1, R = 1, E = R (one expert per rank) and K = E;
* the SM count on hand-worked cases where every step (bounding time per
  token, the larger of read and write SMs, x 1.25, floor 4, even, floor 64
  without overlap, device cap) comes out in round numbers.
"""
import itertools
from fractions import Fraction

import pytest

import oracle


@pytest.mark.parametrize("E,K,R", [(8, 3, 4), (12, 4, 3), (6, 2, 6), (10, 5, 2), (9, 3, 3)])
def test_expected_ranks_brute_force(E, K, R):
    el = E // R
    subsets = list(itertools.combinations(range(E), K))
    mean = Fraction(sum(len({e // el for e in s}) for s in subsets), len(subsets))
    assert oracle.expected_ranks_per_token(E, K, R) == pytest.approx(float(mean), rel=1e-13)


@pytest.mark.parametrize("E,R", [(256, 8), (64, 16), (2048, 1024), (16, 1)])
def test_expected_ranks_closed_forms(E, R):
    assert oracle.expected_ranks_per_token(E, 1, R) == pytest.approx(1.0, rel=1e-13)
    assert oracle.expected_ranks_per_token(E, 8, 1) == pytest.approx(1.0, rel=1e-13)
    assert oracle.expected_ranks_per_token(R, min(R, 8), R) == pytest.approx(min(R, 8), rel=1e-13)
    assert oracle.expected_ranks_per_token(E, E if E <= 32 else 32, R) <= R
    assert oracle.expected_ranks_per_token(16, 16, 4) == pytest.approx(4.0, rel=1e-13)


def test_sm_count_hand_worked():
    # E = R = 8, K = 4: every token reaches exactly g = 4 ranks.  H = 128 bf16:
    # dispatch reads 256 B and writes 1024 B per token; at 1000 GB/s the HBM
    # moves a token in 1.28 ns, so reads need 256/200/1.28 = 1 SM and writes
    # 1024/50/1.28 = 16 SMs; x 1.25 = 20.
    c, n = oracle.theoretical_num_sms(128, 4, 8, 8, 1000.0)
    assert n == pytest.approx(16.0) and c == 20
    assert oracle.theoretical_num_sms(128, 4, 8, 8, 1000.0, prefer_overlap=False)[0] == 64
    assert oracle.theoretical_num_sms(128, 4, 8, 8, 1000.0, device_sms=16)[0] == 16
    # combine: read 1024 B, write 256 B: 1024/200/1.28 = 4 = 256/50/1.28;
    # x 1.25 = 5, rounded up to even = 6
    c, n = oracle.theoretical_num_sms(128, 4, 8, 8, 1000.0, combine=True)
    assert n == pytest.approx(4.0) and c == 6
    # floor of 4: at 100 GB/s the dispatch needs 1.6 SMs -> 2 -> 4
    c, n = oracle.theoretical_num_sms(128, 4, 8, 8, 100.0)
    assert n == pytest.approx(1.6) and c == 4
    # FP8 rows are 128 + 4 bytes: read 256, write 528, at 784 GB/s one token
    # per ns: max(1.28, 10.56) x 1.25 = 13.2 -> 14
    c, n = oracle.theoretical_num_sms(128, 4, 8, 8, 784.0, fp8=True)
    assert n == pytest.approx(10.56) and c == 14
    # combine ignores FP8 (it reads bf16 rows)
    assert oracle.theoretical_num_sms(128, 4, 8, 8, 1000.0, fp8=True, combine=True)[0] == 6
    # 17 SMs x 1.25 = 21.25 -> 22 (ceil, then even)
    c, n = oracle.theoretical_num_sms(128, 4, 8, 8, 1062.5)
    assert n == pytest.approx(17.0) and c == 22
