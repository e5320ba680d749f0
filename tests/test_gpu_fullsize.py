"""Full-size runs of the fragmented, block-seam and adapter-drift workloads in
the launch configuration the library uses for them.

At full depth this random-weight stack amplifies rounding differences (see the
Llama-shaped full-size test), so each run is checked on outputs the oracle can
compute from the inputs alone, plus properties that hold at any size:
  - layer 0's written K/V rows (their inputs are the gathered embedding rows)
    elementwise against the oracle's layer 0;
  - the refreshed rows after layer 0 (X^1, from a run of layer 0 alone)
    elementwise against the oracle's layer 0: they pass through the biased
    attention over the whole cache, the output projection and the MLP, and
    depend on the inputs alone, so no GPU value enters the oracle;
  - every K/V row outside the refreshed set bit-identical to the input cache;
  - the metadata commit bit-exact; every refreshed value finite."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from selective_kv_cache_gb300 import workloads as wl

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup, merge_lora, pack_adapter  # noqa: E402
from helpers import TOL, LazyWeights, assert_close, assert_close_rows, f64, oracle_spec  # noqa: E402


def layer0_oracle(s, seq, rows, alpha, beta, sink_static=False, weights=None):
    """Oracle layer 0 for the selected rows of one sequence."""
    w = s.w
    spec = dataclasses.replace(oracle_spec(w), n_layers=1)
    U = oracle.sorted_positions(rows)
    ids = s.ids[seq].cpu().numpy()
    X_src = np.zeros((w.capacity, w.model.d_model))
    X_src[U] = f64(s.embed[torch.from_numpy(ids[U].astype(np.int64)).to(s.embed.device)])
    W = LazyWeights(weights if weights is not None else s.layers)
    K0 = f64(s.K_in[seq, :1])
    V0 = f64(s.V_in[seq, :1])
    X1, K, V, _, _ = oracle.refresh_packed(spec, W, K0, V0, s.local_mask[seq], s.sink_mask[seq], U, X_src, alpha,
                                           beta, sink_static, n_layers=1)
    return U, K[0], V[0], X1


def run_layer0(s, flags=0):
    """Layer 0 alone on the current selection; returns the refreshed rows X^1.
    It writes only layer 0's selected K/V rows, which a later full refresh
    rewrites before reading them, so the full run's results do not change."""
    s.select()
    s.refresh(0, 1, flags=flags)
    s.sync()
    return f64(s.hidden[:s.n_rows])


def check_untouched(s, seq, layer, rows):
    keep = torch.ones(s.w.capacity, dtype=torch.bool, device=s.K.device)
    keep[torch.from_numpy(np.asarray(rows)).to(s.K.device)] = False
    assert torch.equal(s.K[seq, layer][:, keep], s.K_in[seq, layer][:, keep])
    assert torch.equal(s.V[seq, layer][:, keep], s.V_in[seq, layer][:, keep])


def test_fragmented_packed_and_interval_wise_full_size():
    """282 isolated positions of the 5632-token suffix (about 270 intervals):
    both schedules against the oracle's layer 0, and against each other."""
    w = wl.WORKLOADS["llama8b_frag"]
    a = Setup(w)
    a.K_in, a.V_in = a.K.clone(), a.V.clone()
    b = Setup(w, weights=a.layers, cache=(a.K_in.clone(), a.V_in.clone()))
    b.K_in, b.V_in = a.K_in, a.V_in
    X1_gpu = run_layer0(a)
    a.select()
    a.refresh()
    a.sync()
    n_iv = b.refresh_interval_wise()
    b.sync()
    U, K0, V0, X1 = layer0_oracle(a, 0, a.positions[0], 0.0, 0.0)
    assert_close_rows(X1_gpu, X1, TOL["bf16"], "refreshed rows after layer 0")
    assert n_iv == oracle.intervals(U).shape[0] and n_iv > 250
    Ut = torch.from_numpy(U)
    for s in (a, b):
        assert_close(f64(s.K[0, 0][:, Ut]), K0[:, U], TOL["bf16"], "K layer 0")
        assert_close(f64(s.V[0, 0][:, Ut]), V0[:, U], TOL["bf16"], "V layer 0")
        for layer in (0, 15, 31):
            check_untouched(s, 0, layer, U)
        assert torch.isfinite(s.hidden[:len(U)].float()).all()
    assert_close(f64(b.K[0, 0][:, Ut]), f64(a.K[0, 0][:, Ut]), TOL["bf16"], "packed vs interval-wise K layer 0")
    la, _ = kvr.kvr_read_meta(a.handle, 1, a.words)
    lb, _ = kvr.kvr_read_meta(b.handle, 1, b.words)
    np.testing.assert_array_equal(la, lb)
    a.close()
    b.close()


@pytest.mark.parametrize("sink_static", [False, True])
def test_block_seam_full_size(sink_static):
    """N = 16384 in 8 independently prefilled blocks, T_tau seams (896
    positions, 8 intervals), alpha = -2, beta = -4, Qwen2.5-7B shape (7 query
    heads per K/V head, q/k/v bias)."""
    w = wl.WORKLOADS["qwen7b_seam"]
    s = Setup(w, flags=kvr.KVR_SINK_STATIC if sink_static else 0)
    s.K_in, s.V_in = s.K.clone(), s.V.clone()
    X1_gpu = run_layer0(s)
    rows, ivs = s.select()
    assert rows == 896 and ivs == 8
    s.refresh()
    s.sync()
    U, K0, V0, X1 = layer0_oracle(s, 0, s.positions[0], w.alpha, w.beta, sink_static)
    assert_close_rows(X1_gpu, X1, TOL["bf16"], "refreshed rows after layer 0 (alpha/beta bias, 7 heads per K/V head)")
    Ut = torch.from_numpy(U)
    assert_close(f64(s.K[0, 0][:, Ut]), K0[:, U], TOL["bf16"], "K layer 0")
    assert_close(f64(s.V[0, 0][:, Ut]), V0[:, U], TOL["bf16"], "V layer 0")
    for layer in (0, 13, 27):
        check_untouched(s, 0, layer, U)
    assert torch.isfinite(s.hidden[:rows].float()).all()
    sel = np.zeros(w.capacity, bool)
    sel[U] = True
    local, sink = kvr.kvr_read_meta(s.handle, 1, s.words)
    np.testing.assert_array_equal(local[0], oracle.bitmask_words(s.local_mask[0] & ~sel)[:s.words])
    want_sink = s.sink_mask[0] if sink_static else (s.sink_mask[0] & ~sel)
    np.testing.assert_array_equal(sink[0], oracle.bitmask_words(want_sink)[:s.words])
    s.close()


def test_adapter_drift_full_size():
    """Batch 4 x 32768, rank-16 LoRA on Q and V merged on the GPU; the
    layer-range policy picks layers 10-14, which run over the whole
    24576-token affected suffix from stored boundary states; 492 isolated
    positions per sequence in the other layers."""
    w = wl.WORKLOADS["qwen1p5b_drift"]
    m = w.model
    layers = wl.make_layer_weights(w, "cuda", lora="new")
    # the recovery range comes from the layer-range policy (CacheReforge, Eqs.
    # 8-9): anchors at the old adapter, synthetic sensitivities calibrated on
    # windows [10, 15) at distances 0.8-1.0 x the observed drift
    old = wl.make_layer_weights(w, "cuda", lora="old")
    theta0, theta1 = pack_adapter(old), pack_adapter(layers)
    del old
    d_obs = float((theta1.float() - theta0.float()).norm())
    cal = np.random.default_rng(3)
    s_l = kvr.kvr_policy_sensitivity(m.n_layers, [10] * 40, [5] * 40, d_obs * cal.uniform(0.8, 1.0, 40))
    pol = kvr.kvr_policy_create(m.n_layers, theta0, s_l)
    _, q, (r0, r1) = kvr.kvr_policy_plan(pol, m.n_layers, theta1, kvr.KVR_MOD_V, 10)
    assert (r0, r1) == w.range_layers and np.all(q[10:15] >= 1.0) and np.all(q[15:] == 0.0)
    kvr.kvr_policy_commit(pol, theta1, r0, r1, 1)
    assert kvr.kvr_policy_plan(pol, m.n_layers, theta1, kvr.KVR_MOD_V, 10)[2] == (10, 10)   # now current: reuse
    kvr.kvr_policy_destroy(pol)
    merged = merge_lora(layers, w.model)
    for L in layers:        # the base projections are no longer needed on the device
        L["w_qkv"] = None
    s = Setup(w, weights=merged)
    s.K_in, s.V_in = s.K.clone(), s.V.clone()
    X1_gpu = run_layer0(s)      # the 492 isolated rows per sequence, through layer 0 under the merged adapter
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed(6) * 1000 + 7)
    boundary = torch.empty((w.batch, w.capacity, w.model.d_model), device="cuda", dtype=torch.float32)
    boundary.normal_(0.0, 1.0, generator=g)
    boundary = boundary.to(torch.bfloat16)
    s.refresh_range(boundary, r0, r1)
    # the oracle runs the merged projection as it is (the merge itself is pinned
    # by the LoRA test); the adapter terms are already inside w_qkv
    plain = [{k: v for k, v in L.items() if k not in ("a_q", "b_q", "a_v", "b_v")} for L in merged]
    s.sync()
    full = np.arange(w.suffix_start, w.n_tokens)
    off = 0
    for seq in range(w.batch):
        # layer 0 runs the selected rows only, under the merged adapter
        U, K0, V0, X1 = layer0_oracle(s, seq, s.positions[seq], 0.0, 0.0, weights=plain)
        assert_close_rows(X1_gpu[off:off + len(U)], X1, TOL["bf16"], f"refreshed rows of seq {seq} after layer 0")
        off += len(U)
        Ut = torch.from_numpy(U)
        assert_close(f64(s.K[seq, 0][:, Ut]), K0[:, U], TOL["bf16"], f"K seq {seq} layer 0")
        assert_close(f64(s.V[seq, 0][:, Ut]), V0[:, U], TOL["bf16"], f"V seq {seq} layer 0")
        check_untouched(s, seq, 0, U)
        check_untouched(s, seq, 20, U)
        check_untouched(s, seq, r0, full)          # the range rewrites the whole suffix, nothing else
        changed = (s.K[seq, r0][:, torch.from_numpy(full).cuda()] != s.K_in[seq, r0][:, torch.from_numpy(full).cuda()])
        assert changed.any(dim=-1).float().mean() > 0.99
    assert torch.isfinite(s.hidden[:s.n_rows].float()).all()
    s.close()
