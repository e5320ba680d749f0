"""Pins for the oracle's layer-range policy (CacheReforge: Bounded Recovery
for Stale KV Caches under Evolving Adapters): hand-worked cases of Eq. S4,
Eqs. 6-7 and Eqs. 8-9, and the anchor bookkeeping under repeated updates."""
import numpy as np

from oracle import policy as P


def test_restart_layer_eq_s4():
    N = 28
    assert P.restart_layer(P.MOD_K, 10, N) == 10
    assert P.restart_layer(P.MOD_V, 0, N) == 0
    assert P.restart_layer(P.MOD_Q, 10, N) == 11
    assert P.restart_layer(P.MOD_O, 10, N) == 11
    assert P.restart_layer(P.MOD_MLP, 3, N) == 4
    # a query/output/MLP update in the last layer changes no cached layer: the sentinel N
    assert P.restart_layer(P.MOD_Q, N - 1, N) == N


def test_sensitivity_worked_examples():
    # three layers; conditions (restart, first safe window, distance):
    #   (0, 2, 0.5) labels layers 0, 1; (1, 1, 0.2) labels layer 1; (1, 0, 9.0) is direct reuse
    s = P.sensitivity(3, [0, 1, 1], [2, 1, 0], [0.5, 0.2, 9.0])
    # layer 0: D = {0.5} -> delta = 0.5; layer 1: D = {0.2, 0.5} -> delta = 0.2; layer 2: unlabelled
    np.testing.assert_array_equal(s, [2.0, 5.0, 0.0])
    # the 5 % lower tail: 40 labelled distances 1..40 -> floor(0.05 * 40) = 2 -> the third smallest
    s = P.sensitivity(1, [0] * 40, [1] * 40, list(range(40, 0, -1)))
    assert s[0] == 1.0 / 3.0
    # 19 distances: floor(0.95) = 0 -> the smallest
    s = P.sensitivity(1, [0] * 19, [1] * 19, list(range(1, 20)))
    assert s[0] == 1.0
    # a zero distance is floored at 1e-12
    assert P.sensitivity(1, [0], [1], [0.0])[0] == 1e12


def test_plan_worked_example():
    theta0 = np.zeros(4)
    delta = np.array([2.0, 0.0, 0.0, 0.0])          # ||delta|| = 2
    s = [0.0, 0.1, 0.6, 0.4, 0.0]                    # q = [0, 0.2, 1.2, 0.8, 0]
    pol = P.Policy(s, theta0, 5)
    d, q, rng = pol.plan(theta0 + delta, P.MOD_K, 1)
    np.testing.assert_allclose(d, 2.0)
    np.testing.assert_allclose(q, [0, 0.2, 1.2, 0.8, 0])
    assert rng == (1, 3)                             # b_t = 1 + 2
    # a query update at layer 2: r_KV = 3 and b_t = 3 -> the range replaces no affected K/V: reuse
    assert pol.plan(theta0 + delta, P.MOD_Q, 2)[2] == (2, 2)
    # nothing triggers below threshold: reuse
    assert pol.plan(theta0 + delta / 4, P.MOD_K, 0)[2] == (0, 0)
    # q exactly 1 triggers (q_l >= 1)
    assert P.Policy([0.5], theta0, 1).plan(theta0 + delta, P.MOD_V, 0)[2] == (0, 1)


def test_anchors_track_a_mixed_version_cache():
    """After a bounded recovery only the recomputed layers move their anchors;
    a later update that cancels the first leaves the untouched layers with no
    drift and the recomputed ones with the full displacement."""
    rng = np.random.default_rng(5)
    theta0 = rng.standard_normal(50)
    delta = rng.standard_normal(50)
    pol = P.Policy([1.0] * 6, theta0, 6)
    pol.commit(theta0 + delta, 2, 4, version=1)
    np.testing.assert_array_equal(pol.version, [0, 0, 1, 1, 0, 0])
    d, _, _ = pol.plan(theta0, P.MOD_V, 0)          # the update undoes delta
    np.testing.assert_allclose(d[[0, 1, 4, 5]], 0.0, atol=0)
    np.testing.assert_allclose(d[[2, 3]], np.linalg.norm(delta), rtol=1e-15)
    # consecutive updates accumulate drift against each layer's own anchor
    d2, _, _ = pol.plan(theta0 + 2 * delta, P.MOD_V, 0)
    np.testing.assert_allclose(d2[[0, 1, 4, 5]], 2 * np.linalg.norm(delta), rtol=1e-15)
    np.testing.assert_allclose(d2[[2, 3]], np.linalg.norm(delta), rtol=1e-15)
