"""Oracle: selection bookkeeping (integer work, compared bit-exactly).

Sources (cited by page title and section):
  [BKR]  "Budgeted KV-Cache Repair for Evolving Contexts"
  [KVX]  "kv-cross-attention-reuse" (mixed cache and operator F), Sec. 6

Every function here is pinned by tests/test_oracle_select.py against brute
force on small inputs and against values the pages print.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "budget", "validate_selection", "sorted_positions", "intervals",
    "bitmask_words", "effective_masks", "tile_plan", "pair_count",
    "seam_set", "block_of", "shift_mask",
]


def budget(S: int, b: int) -> int:
    """Exact allowance B(S, b) = min{S, ceil(S*b/100)} for 0 <= b <= 100
    ([BKR] Sec. 7.1, Eq. 3).  Integer ceiling: (S*b + 99) // 100."""
    if not (0 <= b <= 100):
        raise ValueError("budget percent outside [0, 100]")
    return min(S, (S * b + 99) // 100)


def validate_selection(positions, suffix_start: int, n_tokens: int, budget_percent=None):
    """The support is checked for uniqueness, suffix membership and the exact
    budget before execution ([BKR] Sec. 12 and Sec. 7.1: only retained-suffix
    positions are selectable).  Raises ValueError with a reason."""
    p = np.asarray(positions, dtype=np.int64)
    if p.size and (p.min() < suffix_start or p.max() >= n_tokens):
        raise ValueError("position outside the retained suffix")
    if np.unique(p).size != p.size:
        raise ValueError("duplicate position")
    if budget_percent is not None and budget_percent >= 0:
        if p.size != budget(n_tokens - suffix_start, budget_percent):
            raise ValueError("selection size differs from the exact budget")
    return True


def sorted_positions(positions) -> np.ndarray:
    """U = (u_1 < ... < u_B), zero-based ([BKR] Sec. 13.2)."""
    return np.sort(np.asarray(positions, dtype=np.int64))


def intervals(U) -> np.ndarray:
    """Coalesce sorted positions into maximal half-open intervals [a, b)
    ([BKR] Sec. 3.2 and Algorithm 1: sort A, merge adjacent positions)."""
    U = list(int(u) for u in U)
    out = []
    for u in U:
        if out and out[-1][1] == u:
            out[-1][1] = u + 1
        else:
            out.append([u, u + 1])
    return np.array(out, dtype=np.int64).reshape(-1, 2)


def bitmask_words(flags) -> np.ndarray:
    """Bool [n] -> uint32 words, bit b of word w set iff flags[32w + b]."""
    flags = np.asarray(flags, dtype=bool)
    nw = (flags.size + 31) // 32
    words = np.zeros(nw, dtype=np.uint32)
    for i in np.flatnonzero(flags):
        words[i // 32] |= np.uint32(1) << np.uint32(i % 32)
    return words


def effective_masks(local, sink, selected, sink_static=False):
    """Correction masks seen by the refresh's attention.

    [KVX] Sec. 6.4: M_local(j) = 1[type_j = local], M_sink(j) = 1[j in S'];
    physical repair writes back K/V for selected t and sets type_t <- global.
    [BKR] Eq. 21 writes the selected rows before attention, so a selected key
    is fresh whenever it is read: it counts as global and leaves S' at every
    layer of the refresh.  With sink_static the S' penalty stays on refreshed
    sinks too."""
    local = np.asarray(local, dtype=bool)
    sink = np.asarray(sink, dtype=bool)
    selected = np.asarray(selected, dtype=bool)
    loc = local & ~selected
    snk = sink.copy() if sink_static else (sink & ~selected)
    return loc, snk


def tile_plan(U, rows_per_tile: int, keys_per_tile: int) -> np.ndarray:
    """Reusable execution plan ([BKR] Sec. 13.2, Eqs. 23-24): for each query
    tile of consecutive packed rows with first/last positions u_min, u_max,
        n_full  = floor((u_min + 1) / T_k)   complete-prefix K/V tiles
        n_total = ceil((u_max + 1) / T_k)    total K/V tiles touched.
    The pages use T_k = 64; the tile sizes here are parameters so the plan
    matches whichever kernel consumes it.  Rows: (row0, nrows, u_min, u_max,
    n_full, n_total)."""
    U = sorted_positions(U)
    B = U.size
    out = []
    for r0 in range(0, B, rows_per_tile):
        r1 = min(B, r0 + rows_per_tile)
        umin, umax = int(U[r0]), int(U[r1 - 1])
        n_full = (umin + 1) // keys_per_tile
        n_total = -(-(umax + 1) // keys_per_tile)
        out.append((r0, r1 - r0, umin, umax, n_full, n_total))
    return np.array(out, dtype=np.int64).reshape(-1, 6)


def pair_count(U) -> int:
    """M(U) = sum_{u in U} (u + 1) causal query-key pairs per head
    ([BKR] Sec. 13.2, below Eq. 24)."""
    return int(sum(int(u) + 1 for u in U))


def block_of(n_tokens: int, bounds) -> np.ndarray:
    """Block id b_t of each position for half-open spans B_i = x[s_i:e_i)
    ([KVX] Sec. 6.1)."""
    b = np.full(n_tokens, -1, dtype=np.int64)
    for i, (s, e) in enumerate(bounds):
        b[s:e] = i
    return b


def seam_set(bounds, tau: int) -> np.ndarray:
    """Recomputation set T_tau ([KVX] Sec. 6.3).

    Symmetric window at seam B_i | B_{i+1}: the last tau positions of B_i and
    the first tau of B_{i+1} (each clipped to its block).  Asymmetric rule for
    a true prefix B_1: at the seam B_1 | B_2 the trailing tau of B_1 is
    skipped and that allowance goes to the trailing tau of B_m."""
    sel = set()
    m = len(bounds)
    for i in range(m - 1):
        s_i, e_i = bounds[i]
        s_n, e_n = bounds[i + 1]
        tail = set(range(max(s_i, e_i - tau), e_i))
        head = set(range(s_n, min(e_n, s_n + tau)))
        if i == 0:
            tail = set()
        sel |= tail | head
    s_m, e_m = bounds[m - 1]
    sel |= set(range(max(s_m, e_m - tau), e_m))
    return np.array(sorted(sel), dtype=np.int64)


def shift_mask(mask, start: int, d: int):
    """Per-position flags after Shift deletes [start, start + d) ([BKR]
    Sec. 7.1, Eq. 2): a flag stays with its token, so positions below start
    keep theirs, position p >= start takes the flag of old position p + d,
    and the last d positions, now past the end, read False."""
    m = np.asarray(mask, dtype=bool)
    out = np.zeros_like(m)
    out[..., :start] = m[..., :start]
    n_move = m.shape[-1] - start - d
    out[..., start:start + n_move] = m[..., start + d:]
    return out
