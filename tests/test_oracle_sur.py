"""Pins for the oracle's Semantic-Unit Refresh selection (Budgeted KV-Cache
Repair for Evolving Contexts, Sec. 3.2 / 7.3, Eqs. 1/7 and 8): hand-worked
cosines, top-four means, the envelope of Eq. 8 computed by hand, the ranked
admission, and brute force over all windows."""
import math

import numpy as np

from oracle import sur


def test_token_scores_hand_worked():
    # 2-d embeddings: token 0 = (1, 0), 1 = (0, 2), 2 = (3, 4), 3 = (0, 0)
    E = np.array([[1.0, 0.0], [0.0, 2.0], [3.0, 4.0], [0.0, 0.0]])
    r = sur.token_scores(E, suffix_ids=[0, 1, 2, 3], query_ids=[1])
    # cosines with (0, 1): 0, 1 (+0.25: token 1 is in the query), 0.8, 0 (zero norm)
    np.testing.assert_allclose(r, [0.0, 1.25, 0.8, 0.0], atol=1e-15)
    r = sur.token_scores(E, suffix_ids=[2, 0], query_ids=[0, 1])
    np.testing.assert_allclose(r, [0.8, 1.25], atol=1e-15)     # max over the query tokens


def test_unit_scores_top_four_mean():
    r = np.array([0.1, 0.9, 0.3, 0.5, 0.7, 0.2, 0.4, 0.6])
    # units [0, 5) and [5, 8): top four of the first are 0.9 0.7 0.5 0.3; the second has only three
    np.testing.assert_allclose(sur.unit_scores(r, [0, 5, 8]), [0.6, 0.4], atol=1e-15)


def test_envelope_eq8_by_hand():
    r = [0.5, 0.1, 0.9, 0.2]                      # r_max = 0.9
    g = math.exp(-1 / 16)
    u1 = math.exp(-0.4)
    u2 = max(math.exp(-0.8), g * u1)
    u3 = 1.0
    u4 = max(math.exp(-0.7), g * u3)
    np.testing.assert_allclose(sur.envelope(r), [u1, u2, u3, u4], rtol=1e-15)
    assert u2 == g * u1 and u4 == g            # the decayed peak carries forward
    # width 2: sums u1+u2, u2+u3, u3+u4 -> the last is largest
    assert sur.best_window(r, 2) == 2
    # equal sums: the earliest window wins
    assert sur.best_window([0.0, 0.0, 0.0, 0.0], 2) == 0


def test_best_window_brute_force():
    rng = np.random.default_rng(4)
    for _ in range(100):
        n = int(rng.integers(2, 40))
        r = rng.standard_normal(n)
        w = int(rng.integers(1, n + 1))
        u = sur.envelope(r)
        best = max(range(n - w + 1), key=lambda a: (sum(u[a:a + w]), -a))
        assert sur.best_window(r, w) == best


def test_ranked_admission_worked_example():
    # six tokens, units [0, 2) [2, 5) [5, 6); scores chosen so the ranking is unit 1, unit 0, unit 2
    E = np.eye(6)
    # query token 3: cosine 1 for suffix token id 3, 0 otherwise; the bonus adds 0.25
    suffix = [0, 1, 3, 2, 4, 5]
    bounds = [0, 2, 5, 6]
    r = sur.token_scores(E, suffix, [3])
    np.testing.assert_allclose(r, [0, 0, 1.25, 0, 0, 0])
    us = sur.unit_scores(r, bounds)
    assert sur.unit_order(us) == [1, 0, 2]      # ties of units 0 and 2 break by position
    # budget 50 % of 6 = 3: unit 1 (3 tokens) fills it exactly
    np.testing.assert_array_equal(sur.sur_select(E, suffix, [3], bounds, 50, 100), [102, 103, 104])
    # budget 67 % -> ceil(4.02) = 5: unit 1, then unit 0 (2 tokens) fits exactly
    np.testing.assert_array_equal(sur.sur_select(E, suffix, [3], bounds, 67, 100), [100, 101, 102, 103, 104])
    # budget 34 % -> ceil(2.04) = 3 ... 17 % -> 2: unit 1 does not fit: its best width-2 window;
    # envelope over (1.25, 0, 0): u = (1, e^-1/16, e^-2/16) -> the window starting at the peak
    np.testing.assert_array_equal(sur.sur_select(E, suffix, [3], bounds, 17, 100), [102, 103])
    assert len(sur.sur_select(E, suffix, [3], bounds, 0, 100)) == 0
    np.testing.assert_array_equal(sur.sur_select(E, suffix, [3], bounds, 100, 0), np.arange(6))
