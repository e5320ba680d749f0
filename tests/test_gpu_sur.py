"""GPU parity of Semantic-Unit Refresh selection (kvr_sur_select) against the
oracle (Budgeted KV-Cache Repair for Evolving Contexts, Sec. 3.2 / 7.3, Eqs.
1/7 and 8).  Token scores within 2e-5 (fp32 dot products of length d against
float64); selected positions bit-exact wherever the oracle's selection is
stable under score perturbations of that size (the decision is then unique);
the allowance always exact."""
import numpy as np
import pytest
import torch

from oracle import sur as OS
from oracle.select import budget

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300 import workloads as wl  # noqa: E402


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_from_scores(r, bounds, B, suffix_start):
    """Steps 5-9 of the oracle's selection on given token scores."""
    us = OS.unit_scores(r, bounds)
    A = []
    for k in OS.unit_order(us):
        w = B - len(A)
        if w == 0:
            break
        b, e = bounds[k], bounds[k + 1]
        if e - b <= w:
            A.extend(range(b, e))
        else:
            a = OS.best_window(r[b:e], w)
            A.extend(range(b + a, b + a + w))
            break
    return np.array(sorted(suffix_start + i for i in A))


def perturb(r, seed):
    """Scores moved by up to twice the fp32 error; the exact 1.25 of query
    tokens is not subject to rounding and stays."""
    noise = np.random.default_rng(seed).uniform(-4e-5, 4e-5, r.shape)
    return np.where(r == 1.25, r, r + noise)


def run(E, sids, qids, bounds, bp, suffix_start):
    S = len(sids)
    ws = torch.empty(kvr.kvr_sur_workspace_bytes(S, len(qids), E.shape[1], len(bounds) - 1), dtype=torch.uint8,
                     device="cuda")
    pos = torch.full((S,), -7, dtype=torch.int32, device="cuda")
    sc = torch.empty(S, dtype=torch.float32, device="cuda")
    B = kvr.kvr_sur_select(E, torch.from_numpy(sids).cuda(), torch.from_numpy(qids).cuda(),
                           torch.from_numpy(bounds).cuda(), bp, suffix_start, ws, pos, sc)
    kvr.kvr_sur_status(ws)
    return B, pos[:B].cpu().numpy(), f64(sc), pos


@pytest.mark.parametrize("dtype,d,budgets", [(torch.bfloat16, 512, [0, 3, 5, 20, 100]), (torch.float32, 256, [5, 37])])
def test_sur_matches_oracle(dtype, d, budgets):
    vocab, S, Q, start = 1000, 3000, 40, 700
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    E = torch.randn(vocab, d, generator=g, device="cuda").to(dtype)
    rng = np.random.default_rng(6)
    sids = rng.integers(0, vocab, S).astype(np.int32)
    qids = wl.make_query_ids(vocab, Q, 7, sids, overlap=5)
    bounds = wl.make_unit_bounds(S, 8)
    Ew = f64(E)
    r_ref = OS.token_scores(Ew, sids, qids)
    checked = 0
    for bp in budgets:
        B, pos, sc, buf = run(E, sids, qids, bounds, bp, start)
        assert B == budget(S, bp)
        np.testing.assert_allclose(sc, r_ref, atol=2e-5, rtol=0)
        want = OS.sur_select(Ew, sids, qids, bounds, bp, start)
        assert len(pos) == B and np.all(np.diff(pos) > 0) and np.all((pos >= start) & (pos < start + S))
        assert torch.all(buf[B:] == -7)            # nothing written past the allowance
        pert = [oracle_from_scores(perturb(r_ref, k), bounds, B, start) for k in range(6)]
        if all(np.array_equal(p, want) for p in pert):
            np.testing.assert_array_equal(pos, want)
            checked += 1
    assert checked == len(budgets)


def test_sur_fullsize_llama_shape():
    """The Llama-3-8B-shaped refresh: 32000 x 4096 bf16 embeddings, the
    5632-token retained suffix at 2048, a 64-token query, units of 8-128
    tokens, the 5 % budget (282 positions)."""
    vocab, d, S, Q, start = 32000, 4096, 5632, 64, 2048
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    E = torch.randn(vocab, d, generator=g, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(12)
    sids = rng.integers(0, vocab, S).astype(np.int32)
    qids = wl.make_query_ids(vocab, Q, 13, sids, overlap=6)
    bounds = wl.make_unit_bounds(S, 14)
    B, pos, sc, _ = run(E, sids, qids, bounds, 5, start)
    assert B == 282
    Ew = f64(E)
    r_ref = OS.token_scores(Ew, sids, qids)
    np.testing.assert_allclose(sc, r_ref, atol=2e-5, rtol=0)
    want = OS.sur_select(Ew, sids, qids, bounds, 5, start)
    stable = all(np.array_equal(oracle_from_scores(perturb(r_ref, k), bounds, B, start), want) for k in range(6))
    assert stable
    np.testing.assert_array_equal(pos, want)


def test_sur_validation_and_device_checks():
    E = torch.randn(50, 64, device="cuda")
    sids = torch.arange(10, dtype=torch.int32, device="cuda")
    q = torch.tensor([3, 60], dtype=torch.int32, device="cuda")     # 60 is outside the vocabulary
    bounds = torch.tensor([0, 4, 10], dtype=torch.int32, device="cuda")
    ws = torch.empty(kvr.kvr_sur_workspace_bytes(10, 2, 64, 2), dtype=torch.uint8, device="cuda")
    pos = torch.empty(10, dtype=torch.int32, device="cuda")
    kvr.kvr_sur_select(E, sids, q, bounds, 50, 0, ws, pos)
    with pytest.raises(kvr.KvrError) as e:
        kvr.kvr_sur_status(ws)
    assert e.value.status == kvr.KVR_EDEVICE
    kvr.kvr_sur_status(ws)                          # cleared
    with pytest.raises(kvr.KvrError):
        kvr.kvr_sur_select(E, sids, q[:1], bounds, 101, 0, ws, pos)
    with pytest.raises(kvr.KvrError):
        kvr.kvr_sur_select(E, sids, q[:1], bounds, 50, 0, ws[:16], pos)


def test_sur_tensor_core_path_out_of_range_suffix_ids():
    """bf16 embeddings (the tensor-core path, whose prep kernel gathers the
    suffix rows for the scoring projection): suffix ids outside the vocabulary
    are reported (KVR_EDEVICE) and score as zero rows (cosine 0); every other
    token's score matches the oracle's."""
    vocab, d, S, Q = 300, 512, 700, 24
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    E = torch.randn(vocab, d, generator=g, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(12)
    sids = rng.integers(0, vocab, S).astype(np.int32)
    qids = wl.make_query_ids(vocab, Q, 13, sids, overlap=3)
    bad = np.array([5, 131, 600, 699])
    sids[bad] = [-3, vocab, vocab + 77, -1]
    bounds = wl.make_unit_bounds(S, 14)
    ws = torch.empty(kvr.kvr_sur_workspace_bytes(S, Q, d, len(bounds) - 1), dtype=torch.uint8, device="cuda")
    pos = torch.empty(S, dtype=torch.int32, device="cuda")
    sc = torch.empty(S, dtype=torch.float32, device="cuda")
    kvr.kvr_sur_select(E, torch.from_numpy(sids).cuda(), torch.from_numpy(qids).cuda(), torch.from_numpy(bounds).cuda(),
                       5, 0, ws, pos, sc)
    with pytest.raises(kvr.KvrError) as e:
        kvr.kvr_sur_status(ws)
    assert e.value.status == kvr.KVR_EDEVICE
    # the oracle on a table with one zero row appended, the bad ids pointing at it
    Ew = np.concatenate([f64(E), np.zeros((1, d))])
    s_ref = sids.copy()
    s_ref[bad] = vocab
    r_ref = OS.token_scores(Ew, s_ref, qids)
    assert np.all(r_ref[bad] == 0.0)
    np.testing.assert_allclose(f64(sc), r_ref, atol=2e-5, rtol=0)
