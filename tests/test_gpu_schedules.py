"""GPU parity of the interval-wise comparator and of the adapter-drift layer
range (selection switch with carried rows, on-GPU LoRA merge) against the
oracle's definitions of those schedules."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from selective_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup, merge_lora  # noqa: E402
from helpers import TOL, LazyWeights, assert_close, f64, oracle_spec, small_bf16  # noqa: E402


@pytest.mark.parametrize("selection,sink_static", [("isolated", False), ("units", True)])
def test_interval_wise_matches_oracle_and_packed(selection, sink_static):
    """Budgeted KV-Cache Repair, Sec. 7.1 (sequential maximal-interval replay)
    against the oracle's interval schedule; and the packed executor on the same
    inputs agrees with it (Sec. 13.2)."""
    w = small_bf16(selection=selection, alpha=-2.0, beta=-4.0, n_select=60)
    rng = np.random.default_rng(17)
    local = rng.random((1, w.capacity)) < 0.6
    sink = rng.random((1, w.capacity)) < 0.2
    layers = wl.make_layer_weights(w, "cuda")
    flags = kvr.KVR_SINK_STATIC if sink_static else 0
    a = Setup(w, weights=layers, local=local, sink=sink, flags=flags)
    b = Setup(w, weights=layers, local=local, sink=sink, flags=flags)
    Ks0, Vs0 = f64(a.K[0]), f64(a.V[0])
    emb = f64(a.embed)
    X_src = emb[a.ids[0].cpu().numpy()]
    n_iv = a.refresh_interval_wise()
    a.sync()
    U = oracle.sorted_positions(a.positions[0])
    assert n_iv == oracle.intervals(U).shape[0]
    X, K, V, loc2, snk2 = oracle.refresh_interval(oracle_spec(w), LazyWeights(layers), Ks0, Vs0, local[0], sink[0],
                                                  a.positions[0], X_src, w.alpha, w.beta, sink_static)
    assert_close(f64(a.hidden[:len(U)]), X, TOL["bf16"], "interval-wise hidden")
    for l in range(w.model.n_layers):
        assert_close(f64(a.K[0, l][:, torch.from_numpy(U)]), K[l][:, U], TOL["bf16"], f"K layer {l}")
        assert_close(f64(a.V[0, l][:, torch.from_numpy(U)]), V[l][:, U], TOL["bf16"], f"V layer {l}")
    la, sa = kvr.kvr_read_meta(a.handle, 1, a.words)
    np.testing.assert_array_equal(la[0], oracle.bitmask_words(loc2)[:a.words])
    np.testing.assert_array_equal(sa[0], oracle.bitmask_words(snk2)[:a.words])
    # the packed executor on identical inputs
    b.select()
    b.refresh()
    b.sync()
    assert_close(f64(b.hidden[:len(U)]), f64(a.hidden[:len(U)]), TOL["bf16"], "packed vs interval-wise")
    lb, sb_ = kvr.kvr_read_meta(b.handle, 1, b.words)
    np.testing.assert_array_equal(la, lb)
    a.close()
    b.close()


def test_lora_merge_matches_closed_form():
    rng = np.random.default_rng(3)
    n_out, K, r = 640, 256, 16
    W = torch.from_numpy(rng.standard_normal((n_out, K)).astype(np.float32) * 0.02).to(torch.bfloat16).cuda()
    A = torch.from_numpy(rng.standard_normal((r, K)).astype(np.float32) * 0.01).to(torch.bfloat16).cuda()
    B = torch.from_numpy(rng.standard_normal((128, r)).astype(np.float32) * 0.01).to(torch.bfloat16).cuda()
    out = torch.empty_like(W)
    kvr.kvr_lora_merge(W, out, n_out, K, 256, 128, A, B, r, 1.0, kvr.KVR_BF16)
    torch.cuda.synchronize()
    want = f64(W).copy()
    want[256:384] += f64(B) @ f64(A)
    want = oracle.round_bf16(want)
    got = f64(out)
    # one bf16 rounding of an fp32 sum: at most one ulp away from the exact result
    assert np.max(np.abs(got - want) / np.maximum(np.abs(want), 1e-30)) <= 2.0 ** -7
    np.testing.assert_array_equal(got[:256], f64(W)[:256])


def test_adapter_drift_layer_range_matches_oracle():
    """CacheReforge, Bounded Recovery ("Executable restart"): layers [r0, r1)
    over the whole affected suffix from the stored boundary states, the
    selected rows elsewhere; under a merged LoRA on Q and V."""
    m = wl.ModelShape(4, 512, 12, 2, 128, 1024, 1e6, 1e-6, "bf16", True, vocab=1000)
    w = wl.Workload("drift_small", 8, m, 2, 320, 300, 100, 12, selection="isolated", range_layers=(1, 3),
                    lora_rank=16)
    spec = oracle.Spec.of(m)
    base = wl.make_layer_weights(w, "cuda", lora="new")
    old = wl.make_layer_weights(w, "cuda", lora="old")
    merged = merge_lora(base, m)
    emb = wl.make_embeddings(w, "cuda")
    ids = wl.make_token_ids(w, "cuda")
    W_new = LazyWeights(base)
    W_old = [{k: f64(v) if v is not None else None for k, v in L.items()} for L in old]
    rng = np.random.default_rng(9)
    K0 = np.zeros((w.batch, m.n_layers, m.n_kv_heads, w.capacity, m.head_dim))
    V0 = np.zeros_like(K0)
    bnd = np.zeros((w.batch, w.capacity, m.d_model))
    embn = f64(emb)
    idsn = ids.cpu().numpy()
    for b in range(w.batch):
        X_in = embn[idsn[b]][:w.n_tokens].copy()
        dirty = X_in.copy()
        dirty[w.suffix_start:] += 0.5 * rng.standard_normal(dirty[w.suffix_start:].shape)
        _, Ks, Vs, boundary = oracle.prefill(spec, W_old, dirty, return_boundary_at=1)
        K0[b, :, :, :w.n_tokens] = Ks
        V0[b, :, :, :w.n_tokens] = Vs
        bnd[b, :w.n_tokens] = boundary
    Kt = torch.from_numpy(K0).to(torch.bfloat16).cuda()
    Vt = torch.from_numpy(V0).to(torch.bfloat16).cuda()
    s = Setup(w, cache=(Kt.clone(), Vt.clone()), weights=merged)
    s.embed, s.ids = emb, ids
    boundary_t = torch.from_numpy(bnd).to(torch.bfloat16).cuda()
    s.refresh_range(boundary_t, 1, 3)
    s.sync()
    off = 0
    for b in range(w.batch):
        U = oracle.sorted_positions(s.positions[b])
        X, K, V, _, _ = oracle.refresh_range(spec, W_new, f64(Kt[b]), f64(Vt[b]), s.local_mask[b], s.sink_mask[b],
                                             U, embn[idsn[b]], f64(boundary_t[b]), w.suffix_start, w.n_tokens, 1, 3)
        assert_close(f64(s.hidden[off:off + len(U)]), X, TOL["bf16"], f"hidden seq {b}")
        full = np.arange(w.suffix_start, w.n_tokens)
        for l in range(m.n_layers):
            rows = full if 1 <= l < 3 else U
            assert_close(f64(s.K[b, l][:, torch.from_numpy(rows)]), K[l][:, rows], TOL["bf16"], f"K seq {b} layer {l}")
            assert_close(f64(s.V[b, l][:, torch.from_numpy(rows)]), V[l][:, rows], TOL["bf16"], f"V seq {b} layer {l}")
        off += len(U)
    s.close()
