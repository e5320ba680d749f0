"""Model check of the projection kernel's barrier protocol
(selective_kv_cache_gb300/csrc/gemm.cu), run on the CPU.

One persistent CTA walks its items (a feature tile, a row tile, a K range of
kb blocks each); the roles are played out as coroutines under random
interleavings, with TMA landings in any order and tensor-core products
completing in issue order:

  producer   ring of `stages` slots: iteration it (the it-th K block over all
             items) uses slot it % stages; the first `pre` iterations are
             armed up front (the weight tiles go out before the wait for the
             previous kernel), every later one waits for empty[s] (the
             product that read the slot) before it re-arms full[s];
  MMA        per item waits acc_empty[ab] (ab = item parity: the epilogue has
             drained that accumulator), per K block waits full[s], issues and
             commits empty[s]; after the item commits acc_full[ab];
  epilogue   kEpiWarps warps, each waits acc_full[ab], reads its share and
             arrives on acc_empty[ab] (count kEpiWarps).

With overlapping accumulator windows (two windows of more than half the
tensor-memory columns, at both ends), every window holds the shared columns:
the epilogue reads its share of those first and arrives on ovl_free (count
kEpiWarps), then reads the rest; the MMA role waits, before item i's first
product, for ovl_free's completion i - 1 as well as for acc_empty[ab].

The first polls of empty and acc_empty ask for the phase before phase 0
(parity 1 on a fresh barrier), which a fresh barrier reports complete.  The
model asserts that no poll is fooled by a barrier two phases away, that no
barrier is re-armed with a phase open, that a ring slot is refilled only
after its product read it, that an accumulator is overwritten only after
every epilogue warp has read it and, with overlapping windows, that the
shared columns are overwritten only after every epilogue warp has read the
previous item's share of them.
"""
import random

import pytest

K_EPI_WARPS = 12


class Alias(AssertionError):
    pass


class Hazard(AssertionError):
    pass


def simulate(item_kbs, stages, seed, wait_acc_empty=True, ovl=False, wait_ovl=True):
    R = random.Random(seed)
    total = sum(item_kbs)
    pre = min(stages, total)
    done = {}
    arrivals = {}
    fin = {"land": set(), "mma": set(), "drained": set()}
    tma, mma_q = [], []
    acc_reads = {}          # item -> epilogue warps that read it
    shared_reads = {}       # item -> epilogue warps that read its shared columns

    def cnt(b):
        return done.get(b, 0)

    def poll(b, k):
        """Wait for completion number k (0-based) of barrier b; k = -1 is the
        phase before the first, which a fresh barrier reports complete."""
        c = cnt(b)
        if k == -1:
            if c == 0:
                return True
            raise Alias(f"{b}: polling the initial phase with {c} completed")
        if c == k:
            return False
        if c == k + 1:
            return True
        raise Alias(f"{b}: polling phase {k} with {c} completed")

    def check(cond, what):
        if not cond:
            raise Hazard(what)

    def producer():
        # up-front arming of the first `pre` iterations
        for it in range(pre):
            check(cnt(("full", it % stages)) == it // stages, "full re-armed with a phase open")
            tma.append(it)
            yield
        for it in range(pre, total):
            s = it % stages
            while not poll(("empty", s), it // stages - 1):
                yield
            check(it - stages in fin["mma"], "ring slot refilled before its product read it")
            check(cnt(("full", s)) == it // stages, "full re-armed with a phase open")
            tma.append(it)
            yield

    def mma():
        it = 0
        for item, kbs in enumerate(item_kbs):
            ab = item & 1
            if wait_acc_empty:
                while not poll(("acc_empty", ab), (item >> 1) - 1):
                    yield
            if ovl and wait_ovl and item > 0:
                while not poll(("ovl_free",), item - 1):
                    yield
            check(item < 2 or acc_reads.get(item - 2, 0) == K_EPI_WARPS,
                  "accumulator overwritten before the epilogue read it")
            check(not ovl or item < 1 or shared_reads.get(item - 1, 0) == K_EPI_WARPS,
                  "shared columns overwritten before the epilogue read them")
            for _ in range(kbs):
                s = it % stages
                while not poll(("full", s), it // stages):
                    yield
                check(it in fin["land"], "product before its operands landed")
                mma_q.append(("kb", it))
                it += 1
                yield
            mma_q.append(("acc", item))
            yield

    def epi_warp(w):
        for item in range(len(item_kbs)):
            ab = item & 1
            while not poll(("acc_full", ab), item >> 1):
                yield
            check(item in fin["drained"], "accumulator read before its products finished")
            if ovl:
                shared_reads[item] = shared_reads.get(item, 0) + 1
                yield
                key = ("ovl_free",)
                arrivals[key] = arrivals.get(key, 0) + 1
                if arrivals[key] == K_EPI_WARPS:
                    arrivals[key] = 0
                    done[key] = cnt(key) + 1
                yield
            acc_reads[item] = acc_reads.get(item, 0) + 1
            yield
            key = ("acc_empty", ab)
            arrivals[key] = arrivals.get(key, 0) + 1
            if arrivals[key] == K_EPI_WARPS:
                arrivals[key] = 0
                done[key] = cnt(key) + 1
            yield

    roles = [producer(), mma()] + [epi_warp(w) for w in range(K_EPI_WARPS)]
    live = [True] * len(roles)
    for _ in range(2000000):
        if not (any(live) or tma or mma_q):
            return
        opts = [("role", i) for i, a in enumerate(live) if a]
        opts += [("tma", None)] * bool(tma) + [("mma", None)] * bool(mma_q)
        kind, i = R.choice(opts)
        if kind == "role":
            try:
                next(roles[i])
            except StopIteration:
                live[i] = False
        elif kind == "tma":
            it = tma.pop(R.randrange(len(tma)))
            fin["land"].add(it)
            done[("full", it % stages)] = cnt(("full", it % stages)) + 1
        else:
            what, x = mma_q.pop(0)
            if what == "kb":
                fin["mma"].add(x)
                done[("empty", x % stages)] = cnt(("empty", x % stages)) + 1
            else:
                fin["drained"].add(x)
                done[("acc_full", x & 1)] = cnt(("acc_full", x & 1)) + 1
    raise AssertionError("no progress: deadlock")


@pytest.mark.parametrize("stages", [3, 4, 8])
def test_protocol_has_no_alias_deadlock_or_overwrite(stages):
    R = random.Random(stages)
    for seed in range(150):
        items = [R.randint(1, 6) for _ in range(R.randint(1, 6))]
        simulate(items, stages, seed)


def test_fewer_blocks_than_stages():
    """A CTA whose items hold fewer K blocks than the ring has slots arms
    only those up front."""
    for seed in range(200):
        simulate([1], 3, seed)
        simulate([2], 8, seed)
        simulate([1, 1, 1], 4, seed)


def test_accumulator_reuse_without_its_wait_is_caught():
    hits = 0
    for seed in range(200):
        try:
            simulate([1, 1, 1, 1, 1], 3, seed, wait_acc_empty=False)
        except (Hazard, Alias):
            hits += 1
    assert hits > 0


@pytest.mark.parametrize("stages", [3, 4, 8])
def test_overlapping_windows_have_no_alias_deadlock_or_overwrite(stages):
    R = random.Random(100 + stages)
    for seed in range(150):
        items = [R.randint(1, 6) for _ in range(R.randint(1, 6))]
        simulate(items, stages, seed, ovl=True)


def test_shared_columns_without_their_wait_are_caught():
    hits = 0
    for seed in range(200):
        try:
            simulate([1, 1, 1, 1, 1], 4, seed, ovl=True, wait_ovl=False)
        except (Hazard, Alias):
            hits += 1
    assert hits > 0
