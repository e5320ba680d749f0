"""Oracle: the layer-range policy of "CacheReforge: Bounded Recovery for Stale
KV Caches under Evolving Adapters" (Methodology: Layerwise Risk, Eqs. 6-7;
Runtime risk and range selection, Eqs. 8-9; Cache and anchor updates;
supplementary Eq. S4).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in
float64; the adapter is one flat parameter vector theta.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["MOD_Q", "MOD_K", "MOD_V", "MOD_O", "MOD_MLP", "restart_layer", "sensitivity", "drift",
           "plan", "Policy"]

MOD_Q, MOD_K, MOD_V, MOD_O, MOD_MLP = range(5)


def restart_layer(module: int, s: int, n_layers: int) -> int:
    """r_KV(m, s) (Eq. S4): a key or value update changes the cache written
    at layer s itself; a query, output or MLP update changes the layer's
    output but not the K/V already written there, so the first cache layer
    that can change is s + 1 (capped at the sentinel N)."""
    if module in (MOD_K, MOD_V):
        return s
    if module in (MOD_Q, MOD_O, MOD_MLP):
        return min(s + 1, n_layers)
    raise ValueError("unknown module")


def sensitivity(n_layers: int, restart, window, dist):
    """Eqs. 6-7.  Label y_{i,l} = 1 when restart_i <= l < restart_i + h*_i;
    D_l collects the distances of the labelled conditions; delta_l is the
    order statistic just past the allowed 5 % lower tail,
    d_(floor(0.05 n_l) + 1) in 1-based terms, floored at 1e-12;
    s_l = 1 / delta_l, or 0 when no condition labels the layer."""
    s = np.zeros(n_layers)
    for l in range(n_layers):
        D = sorted(float(d) for r, h, d in zip(restart, window, dist) if r <= l < r + h)
        if not D:
            continue
        k = math.floor(0.05 * len(D))      # 0-based index of d_(floor(0.05 n) + 1)
        s[l] = 1.0 / max(D[k], 1e-12)
    return s


def drift(theta_t, anchors):
    """d_l(t) = ||theta_t - theta_l^anchor||_2 for every layer (Eq. 8)."""
    theta_t = np.asarray(theta_t, dtype=np.float64)
    return np.array([np.linalg.norm(theta_t - np.asarray(a, dtype=np.float64)) for a in anchors])


def plan(s, anchors, theta_t, module: int, update_layer: int):
    """Risk q_l = s_l d_l; layer l triggers when q_l >= 1; b_t = 1 + max of the
    triggered layers (Eq. 9); the recovery range is [r, b_t) from the
    executable restart r = update_layer.  No trigger, or a range ending at or
    before r_KV (it would replace no affected K/V state), is direct reuse:
    the empty range [r, r).  Returns (d, q, (begin, end))."""
    N = len(anchors)
    d = drift(theta_t, anchors)
    q = np.asarray(s, dtype=np.float64) * d
    trig = np.flatnonzero(q >= 1.0)
    r = update_layer
    if trig.size == 0:
        return d, q, (r, r)
    b = int(trig.max()) + 1
    if b <= restart_layer(module, update_layer, N):
        return d, q, (r, r)
    return d, q, (r, b)


class Policy:
    """Per-layer anchors and versions ("Cache and anchor updates"): after a
    range is recomputed under theta_t only its layers take theta_t as their
    anchor; the others keep their older anchors."""

    def __init__(self, s, theta0, n_layers: int):
        self.s = np.asarray(s, dtype=np.float64)
        self.anchors = [np.asarray(theta0, dtype=np.float64).copy() for _ in range(n_layers)]
        self.version = np.zeros(n_layers, dtype=np.int64)

    def plan(self, theta_t, module: int, update_layer: int):
        return plan(self.s, self.anchors, theta_t, module, update_layer)

    def commit(self, theta_t, begin: int, end: int, version: int):
        for l in range(begin, end):
            self.anchors[l] = np.asarray(theta_t, dtype=np.float64).copy()
            self.version[l] = version
