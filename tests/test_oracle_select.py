"""Pins for the oracle's integer bookkeeping (CPU only).

Each function is checked against something other than itself: values the
pages print (tests/golden/pages_worked_examples.json), brute force over
Python sets and ints, or closed forms.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "pages_worked_examples.json")))


def test_budget_printed_examples():
    for c in GOLDEN["budgets"]["cases"]:
        assert oracle.budget(c["S"], c["b"]) == c["B"]


def test_budget_closed_form_sweep():
    for S in [0, 1, 7, 99, 100, 101, 5632, 24576]:
        for b in range(0, 101):
            want = min(S, math.ceil(S * b / 100)) if S * b % 100 else min(S, S * b // 100)
            assert oracle.budget(S, b) == want
    assert oracle.budget(5632, 5) == 282
    assert oracle.budget(24576, 2) == 492
    with pytest.raises(ValueError):
        oracle.budget(10, 101)


def test_validate_selection_rejects():
    oracle.validate_selection([5, 7, 9], 5, 10)
    with pytest.raises(ValueError):
        oracle.validate_selection([4, 7], 5, 10)          # in the prefix
    with pytest.raises(ValueError):
        oracle.validate_selection([5, 10], 5, 10)         # past the end
    with pytest.raises(ValueError):
        oracle.validate_selection([5, 7, 7], 5, 10)       # duplicate
    with pytest.raises(ValueError):
        oracle.validate_selection([5, 6], 0, 100, budget_percent=5)  # needs 5
    oracle.validate_selection([5, 6, 7, 8, 9], 0, 100, budget_percent=5)


def _intervals_brute(U):
    s = set(int(u) for u in U)
    out = []
    for u in sorted(s):
        if u - 1 not in s:
            b = u
            while b in s:
                b += 1
            out.append([u, b])
    return out


def test_intervals_brute_force():
    rng = np.random.default_rng(1)
    for trial in range(200):
        n = int(rng.integers(1, 300))
        k = int(rng.integers(0, n + 1))
        U = np.sort(rng.choice(n, size=k, replace=False))
        got = oracle.intervals(U).tolist()
        assert got == _intervals_brute(U)
        assert sum(b - a for a, b in got) == k


def test_bitmask_words_brute_force():
    rng = np.random.default_rng(2)
    for n in [1, 31, 32, 33, 100, 1024, 7680]:
        f = rng.random(n) < 0.3
        words = oracle.bitmask_words(f)
        big = sum(1 << i for i in range(n) if f[i])
        for w in range(words.size):
            assert int(words[w]) == (big >> (32 * w)) & 0xFFFFFFFF


def test_effective_masks_truth_table():
    local = np.array([0, 0, 1, 1, 0, 0, 1, 1], bool)
    sink = np.array([0, 1, 0, 1, 0, 1, 0, 1], bool)
    sel = np.array([0, 0, 0, 0, 1, 1, 1, 1], bool)
    loc, snk = oracle.effective_masks(local, sink, sel)
    assert loc.tolist() == [0, 0, 1, 1, 0, 0, 0, 0]
    assert snk.tolist() == [0, 1, 0, 1, 0, 0, 0, 0]
    loc, snk = oracle.effective_masks(local, sink, sel, sink_static=True)
    assert snk.tolist() == sink.tolist()


def test_pair_count_printed_examples():
    # any 64-position support centred on N/2 - 1/2 gives the printed counts
    for c in GOLDEN["pair_counts"]["cases"]:
        N, B = c["n_tokens"], c["B"]
        lo = N // 2 - B // 2
        assert oracle.pair_count(range(lo, lo + B)) == c["M"]
        # R = 4 and R = 16 intervals with the same mean position (Sec. 13.3:
        # the count is identical across R)
        for R in (4, 16):
            w = B // R
            starts = [lo + i * 3 * w - (R - 1) * w for i in range(R)]
            U = [s + t for s in starts for t in range(w)]
            assert len(set(U)) == B
            assert abs(np.mean(U) - (N / 2 - 0.5)) < 1e-9
            assert oracle.pair_count(U) == c["M"]


def test_pair_bound_eq18():
    for c in GOLDEN["pair_bound"]["cases"]:
        assert min(1.0, 2 * c["B"] / c["S"]) == pytest.approx(c["bound"])
    rng = np.random.default_rng(3)
    for _ in range(300):
        P = int(rng.integers(0, 500))
        S = int(rng.integers(1, 500))
        B = int(rng.integers(0, S + 1))
        A = rng.choice(np.arange(1, S + 1), size=B, replace=False)   # 1-based suffix indices
        U = P + A - 1
        full = S * P + S * (S + 1) / 2
        m = oracle.pair_count(U)
        assert m == sum(P + int(i) for i in A)
        assert m <= B * (P + S) - B * (B - 1) / 2 + 1e-9
        assert m / full <= min(1.0, 2 * B / S) + 1e-12


def test_tile_plan_brute_force():
    rng = np.random.default_rng(4)
    for _ in range(100):
        N = int(rng.integers(1, 3000))
        B = int(rng.integers(1, min(N, 400) + 1))
        U = np.sort(rng.choice(N, size=B, replace=False))
        Tq = int(rng.choice([16, 18, 21, 32, 128]))
        Tk = int(rng.choice([64, 128]))
        plan = oracle.tile_plan(U, Tq, Tk)
        assert plan[:, 1].sum() == B
        for (r0, nr, umin, umax, nf, nt) in plan:
            rows = U[r0:r0 + nr]
            n_tiles = (N + Tk - 1) // Tk + 1
            full = [t for t in range(n_tiles) if all(j <= u for u in rows for j in range(t * Tk, (t + 1) * Tk))]
            touched = [t for t in range(n_tiles) if any(t * Tk <= u for u in rows)]
            assert umin == rows.min() and umax == rows.max()
            assert nf == len(full) and full == list(range(nf))
            assert nt == len(touched) and touched == list(range(nt))


def test_blocks_printed_example():
    g = GOLDEN["blocks"]
    b = oracle.block_of(1000, [(g["s1"], g["e1"]), (g["e1"], 1000)])
    members = np.flatnonzero(b == 0)
    assert members[0] == g["first"] and members[-1] == g["last"] and members.size == g["size"]


def _seam_brute(n_blocks, size, tau):
    # membership by distance to the block edges, per the rule's wording
    out = []
    for t in range(n_blocks * size):
        i, off = divmod(t, size)
        head = i >= 1 and off < tau                          # first tau of B_2..B_m
        tail = (1 <= i < n_blocks - 1) and off >= size - tau  # last tau of B_2..B_{m-1}
        last = i == n_blocks - 1 and off >= size - tau       # reallocated tail of B_m
        if head or tail or last:
            out.append(t)
    return out


def test_seam_set_brute_force_and_count():
    for (m, size, tau) in [(8, 2048, 64), (3, 100, 10), (4, 50, 30), (2, 64, 64)]:
        bounds = [(i * size, (i + 1) * size) for i in range(m)]
        got = oracle.seam_set(bounds, tau).tolist()
        assert got == _seam_brute(m, size, tau)
    bounds = [(i * 2048, (i + 1) * 2048) for i in range(8)]
    T = oracle.seam_set(bounds, 64)
    assert T.size == 896
    assert oracle.intervals(T).shape[0] == 8


def test_shift_mask_worked_example_and_brute_force():
    """Flags move with their tokens under Shift (Budgeted KV-Cache Repair,
    Sec. 7.1, Eq. 2).  Worked by hand: flags at 1, 3, 5, 8, 9 of ten
    positions; deleting [2, 5) drops 3 and moves 5 -> 2, 8 -> 5, 9 -> 6."""
    m = np.isin(np.arange(10), [1, 3, 5, 8, 9])
    np.testing.assert_array_equal(np.flatnonzero(oracle.shift_mask(m, 2, 3)), [1, 2, 5, 6])
    rng = np.random.default_rng(71)
    for _ in range(50):
        N = int(rng.integers(1, 200))
        start = int(rng.integers(0, N))
        d = int(rng.integers(0, N - start + 1))
        m = rng.random((2, N)) < 0.4
        want = np.zeros_like(m)
        for b in range(2):
            kept = [m[b, p] for p in range(N) if not (start <= p < start + d)]
            want[b, :len(kept)] = kept
        np.testing.assert_array_equal(oracle.shift_mask(m, start, d), want)
