"""Oracle: Semantic-Unit Refresh selection ("Budgeted KV-Cache Repair for
Evolving Contexts", Sec. 3.2 and Sec. 7.3, Eqs. 1/7 and 8, and the ranked
allocation of Algorithm 1).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in
float64.  Segmenting text into units is outside this oracle: units come in as
a partition of the suffix.
"""
from __future__ import annotations

import math

import numpy as np

from .select import budget

__all__ = ["token_scores", "unit_scores", "unit_order", "envelope", "best_window", "sur_select"]


def token_scores(E, suffix_ids, query_ids):
    """Eq. 1/7: r_i = max_j <E(s_i), E(q_j)> / (||E(s_i)|| ||E(q_j)||)
    + 0.25 * 1[s_i occurs in q].  A zero-norm row has cosine 0.  A token that
    occurs in the query meets its own embedding, whose cosine is exactly 1,
    the largest a cosine can be: its score is exactly 1.25 (floating-point
    dot products would put it a rounding away from 1 and turn the pages' tie
    rule, earlier position first, into noise)."""
    E = np.asarray(E, dtype=np.float64)
    s = E[np.asarray(suffix_ids)]
    q = E[np.asarray(query_ids)]
    ns = np.linalg.norm(s, axis=1)
    nq = np.linalg.norm(q, axis=1)
    sn = np.divide(s, ns[:, None], out=np.zeros_like(s), where=ns[:, None] > 0)
    qn = np.divide(q, nq[:, None], out=np.zeros_like(q), where=nq[:, None] > 0)
    r = (sn @ qn.T).max(axis=1)
    qset = set(int(x) for x in np.asarray(query_ids))
    in_q = np.array([int(x) in qset for x in np.asarray(suffix_ids)], dtype=bool)
    return np.where(in_q, 1.25, r)


def unit_scores(r, bounds):
    """The mean of each unit's four largest token scores (all of them when
    the unit is shorter)."""
    out = []
    for k in range(len(bounds) - 1):
        v = np.sort(np.asarray(r[bounds[k]:bounds[k + 1]], dtype=np.float64))[::-1]
        out.append(float(np.mean(v[:4])))
    return np.array(out)


def unit_order(us):
    """Units ranked by score, higher first; an earlier position breaks ties."""
    return sorted(range(len(us)), key=lambda k: (-us[k], k))


def envelope(r_unit):
    """Eq. 8 over one unit's tokens in order: u_0 = 0,
    u_t = max(exp(r_t - r_max), exp(-1/16) u_{t-1})."""
    r_unit = np.asarray(r_unit, dtype=np.float64)
    rmax = float(np.max(r_unit))
    u = np.zeros(len(r_unit))
    prev = 0.0
    for t, rt in enumerate(r_unit):
        prev = max(math.exp(rt - rmax), math.exp(-1.0 / 16.0) * prev)
        u[t] = prev
    return u


def best_window(r_unit, w: int) -> int:
    """Offset of the width-w window with the largest envelope sum; the
    earliest maximiser wins."""
    u = envelope(r_unit)
    sums = [float(np.sum(u[a:a + w])) for a in range(len(u) - w + 1)]
    return int(np.argmax(sums))     # argmax returns the first maximiser


def sur_select(E, suffix_ids, query_ids, bounds, budget_percent: int, suffix_start: int):
    """Algorithm 1, steps 1 and 4-9, on a given unit partition: visit units in
    ranked order; a unit that fits the remaining allowance w is taken whole;
    otherwise its best width-w window is taken and the allowance is full.
    Returns the sorted global positions."""
    S = len(suffix_ids)
    B = budget(S, budget_percent)
    r = token_scores(E, suffix_ids, query_ids)
    us = unit_scores(r, bounds)
    A = []
    for k in unit_order(us):
        w = B - len(A)
        if w == 0:
            break
        b, e = bounds[k], bounds[k + 1]
        if e - b <= w:
            A.extend(range(b, e))
        else:
            a = best_window(r[b:e], w)
            A.extend(range(b + a, b + a + w))
            break
    return np.array(sorted(suffix_start + i for i in A), dtype=np.int64)
