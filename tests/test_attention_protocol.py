"""Model check of the tensor-core attention kernel's barrier protocol
(selective_kv_cache_gb300/csrc/attn_tc.cu), run on the CPU.

The kernel's five roles are played out as coroutines under random
interleavings, with TMA landings in any order and tensor-core products
completing in issue order per issuing thread:

  producer   steps t = 0..n: K_t and V_{t-1} on kv_full[t % KS]; before step
             t >= KS it waits for the slot's previous phase, for S_{t-KS}
             (s_full) and, for t >= KS + 1, for the PV product of tile
             t - 1 - KS;
  QK issuer  S_j = Q K_j^T into score buffer j % SB once step j has landed
             and (j >= SB) the PV product of tile j - SB is done;
  PV issuer  O += P_j V_j once P_j (p_full[j & 3]) and step j + 1 are there;
  softmax    waits for S_j, sometimes for the previous PV (an O rescale),
             writes P_j over S_j; at the end waits for the last PV.

KS (ring stages) and SB (score buffers) are the kernel's kStages and kSBufs:
3 and 3; the shallower 2 and 2 (a 64-key, two-CTAs-per-SM form, measured
slower) is checked too.
An mbarrier poll succeeds when the barrier's completed-phase count has the
other parity than the one asked for, so a waiter that falls two phases
behind, or polls a phase two ahead, would be fooled: the model asserts that
never happens, that no barrier is re-armed with a phase still open, and that
no shared-memory slot or tensor-memory buffer is overwritten while a product
or the softmax still reads it.  The variant without the producer's wait for
S_{t-KS} on the last (K-less) step is shown to alias (at KS = 3), which is
why that wait is unconditional in the kernel.
"""
import random

import pytest


class Alias(AssertionError):
    pass


def simulate(n, seed, wait_s_on_last_step=True, KS=3, SB=3):
    """KS: K and V ring stages; SB: score buffers (the kernel's kStages and
    kSBufs)."""
    R = random.Random(seed)
    done = {}                    # barrier -> completed phases
    fin = {"QK": set(), "PV": set(), "P": set(), "land": set()}
    tma, qk_q, pv_q = [], [], []

    def count(b):
        return done.get(b, 0)

    def poll(b, k):
        c = count(b)
        if c == k:
            return False
        if c == k + 1:
            return True
        raise Alias(f"{b}: polling phase {k} with {c} completed")

    def producer():
        for t in range(n + 1):
            if t >= KS:
                while not poll(("kv", t % KS), (t - KS) // KS):
                    yield
                if wait_s_on_last_step or t < n:
                    while not poll(("s", (t - KS) % SB), (t - KS) // SB):
                        yield
                if t >= KS + 1:
                    while not poll(("o", (t - 1 - KS) & 3), (t - 1 - KS) >> 2):
                        yield
            assert count(("kv", t % KS)) == t // KS, "barrier re-armed with a phase open"
            if KS <= t < n:
                assert t - KS in fin["QK"], "K slot overwritten before its product read it"
            if t >= KS + 1:
                assert t - 1 - KS in fin["PV"], "V slot overwritten before its product read it"
            tma.append(t)
            yield

    def qk_issuer():
        for j in range(n):
            while not poll(("kv", j % KS), j // KS):
                yield
            if j >= SB:
                while not poll(("o", (j - SB) & 3), (j - SB) >> 2):
                    yield
                assert j - SB in fin["PV"] and j - SB in fin["P"], "score buffer reused too early"
            qk_q.append(j)
            yield

    def pv_issuer():
        for j in range(n):
            while not poll(("p", j & 3), j >> 2):
                yield
            while not poll(("kv", (j + 1) % KS), (j + 1) // KS):
                yield
            assert j in fin["P"] and j + 1 in fin["land"]
            pv_q.append(j)
            yield

    def softmax():
        for j in range(n):
            while not poll(("s", j % SB), j // SB):
                yield
            assert j in fin["QK"]
            if j > 0 and R.random() < 0.3:   # an O rescale waits for the previous PV
                while not poll(("o", (j - 1) & 3), (j - 1) >> 2):
                    yield
            assert j < SB or j - SB in fin["PV"], "P written over a P still being read"
            fin["P"].add(j)
            done[("p", j & 3)] = count(("p", j & 3)) + 1
            yield
        if n:
            while not poll(("o", (n - 1) & 3), (n - 1) >> 2):
                yield

    roles = [producer(), qk_issuer(), pv_issuer(), softmax()]
    live = [True] * len(roles)
    for _ in range(200000):
        if not (any(live) or tma or qk_q or pv_q):
            return
        opts = [("role", i) for i, a in enumerate(live) if a]
        opts += [("tma", None)] * bool(tma) + [("qk", None)] * bool(qk_q) + [("pv", None)] * bool(pv_q)
        kind, i = R.choice(opts)
        if kind == "role":
            try:
                next(roles[i])
            except StopIteration:
                live[i] = False
        elif kind == "tma":
            t = tma.pop(R.randrange(len(tma)))
            fin["land"].add(t)
            done[("kv", t % KS)] = count(("kv", t % KS)) + 1
        elif kind == "qk":
            j = qk_q.pop(0)
            fin["QK"].add(j)
            done[("s", j % SB)] = count(("s", j % SB)) + 1
        else:
            j = pv_q.pop(0)
            fin["PV"].add(j)
            done[("o", j & 3)] = count(("o", j & 3)) + 1
    raise AssertionError("no progress: deadlock")


@pytest.mark.parametrize("n", list(range(0, 12)))
@pytest.mark.parametrize("KS,SB", [(2, 2), (3, 3)])
def test_protocol_has_no_alias_deadlock_or_overwrite(n, KS, SB):
    """(3, 3) is the kernel's depth; (2, 2) the shallower form the same
    protocol also supports."""
    for seed in range(400):
        simulate(n, seed, KS=KS, SB=SB)


def test_last_step_without_score_wait_aliases():
    """Re-arming the K-less last step after only its slot's landing lets the
    barrier run two phases ahead of the QK issuer (seen at three tiles)."""
    hits = 0
    for seed in range(600):
        try:
            simulate(3, seed, wait_s_on_last_step=False, KS=3, SB=3)
        except Alias:
            hits += 1
    assert hits > 0
