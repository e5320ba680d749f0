"""GPU parity of the packed refresh through the C ABI against the float64
oracle: refreshed hidden rows and written-back K/V within the stated
tolerance, every unselected K/V row bit-identical, metadata bit-exact."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from selective_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup  # noqa: E402
from helpers import TOL, LazyWeights, assert_close, assert_close_rows, f64, oracle_spec, small_bf16  # noqa: E402


def run_and_compare(s: Setup, W_oracle, Ks0, Vs0, X_src_seqs, tol, sink_static=False, check_layers=None):
    """Refresh on the GPU, then the oracle per sequence; compare."""
    w = s.w
    spec = oracle_spec(w)
    K_in = s.K.clone()
    V_in = s.V.clone()
    s.select()
    s.refresh()
    s.sync()
    worst = {}
    off = 0
    local_after, sink_after = kvr.kvr_read_meta(s.handle, w.batch, s.words)
    for seq, pos in enumerate(s.positions):
        n = len(pos)
        U = oracle.sorted_positions(pos)
        X, K, V, loc2, snk2 = oracle.refresh_packed(
            spec, W_oracle, Ks0[seq], Vs0[seq], s.local_mask[seq], s.sink_mask[seq], pos, X_src_seqs[seq],
            w.alpha, w.beta, sink_static)
        worst["hidden"] = max(worst.get("hidden", 0), assert_close(f64(s.hidden[off:off + n]), X, tol, "hidden"))
        layers = range(w.model.n_layers) if check_layers is None else check_layers
        for l in layers:
            Kg = f64(s.K[seq, l][:, torch.from_numpy(U)])
            Vg = f64(s.V[seq, l][:, torch.from_numpy(U)])
            worst["K"] = max(worst.get("K", 0), assert_close(Kg, K[l][:, U], tol, f"K layer {l}"))
            worst["V"] = max(worst.get("V", 0), assert_close(Vg, V[l][:, U], tol, f"V layer {l}"))
        # unselected rows: bit-identical to the input cache
        keep = torch.ones(w.capacity, dtype=torch.bool, device=s.K.device)
        keep[torch.from_numpy(U).to(s.K.device)] = False
        assert torch.equal(s.K[seq][:, :, keep], K_in[seq][:, :, keep])
        assert torch.equal(s.V[seq][:, :, keep], V_in[seq][:, :, keep])
        np.testing.assert_array_equal(local_after[seq], oracle.bitmask_words(loc2)[:s.words])
        np.testing.assert_array_equal(sink_after[seq], oracle.bitmask_words(snk2)[:s.words])
        off += n
    return worst


def test_tiny_fp32_against_oracle_prefill_cache():
    """Tiny fp32 workload: stale cache from the oracle's prefill of the dirty
    sequence, refresh with the clean inputs, tolerance 1e-4."""
    w = wl.WORKLOADS["tiny"]
    spec = oracle_spec(w)
    layers_cpu = wl.make_layer_weights(w, "cpu")
    W = [{k: f64(v) for k, v in L.items()} for L in layers_cpu]
    dirty = f64(wl.make_hidden_inputs(w, "cpu", dirty=True))[0]
    clean = f64(wl.make_hidden_inputs(w, "cpu"))[0]
    _, Ks, Vs = oracle.prefill(spec, W, dirty)
    Kt = torch.from_numpy(Ks[None]).float().cuda().contiguous()
    Vt = torch.from_numpy(Vs[None]).float().cuda().contiguous()
    layers = [{k: (v.cuda() if v is not None else None) for k, v in L.items()} for L in layers_cpu]
    s = Setup(w, cache=(Kt, Vt), weights=layers)
    worst = run_and_compare(s, W, Ks[None], Vs[None], [clean], TOL["f32"])
    s.close()
    print("tiny worst scaled errors", worst)


@pytest.mark.parametrize("selection,alpha,beta,sink_static", [
    ("units", 0.0, 0.0, False),
    ("units", -2.0, -4.0, False),
    ("isolated", -2.0, -4.0, True),
    ("isolated", 1.0, -3.0, False),
])
def test_bf16_small_against_oracle(selection, alpha, beta, sink_static):
    """Small bf16 model (head_dim 128, 4 query heads per K/V head, q/k/v
    bias), several query tiles with a ragged tail, random local/sink masks."""
    w = small_bf16(selection=selection, alpha=alpha, beta=beta)
    rng = np.random.default_rng(11)
    local = rng.random((1, w.capacity)) < 0.6
    sink = rng.random((1, w.capacity)) < 0.2
    layers = wl.make_layer_weights(w, "cuda")
    s = Setup(w, weights=layers, local=local, sink=sink,
              flags=kvr.KVR_SINK_STATIC if sink_static else 0)
    W = LazyWeights(layers)
    Ks0, Vs0 = f64(s.K), f64(s.V)
    emb = f64(s.embed)
    ids = s.ids.cpu().numpy()
    X_src = [emb[ids[b]] for b in range(w.batch)]
    worst = run_and_compare(s, W, Ks0, Vs0, X_src, TOL["bf16"], sink_static=sink_static)
    s.close()
    print(selection, alpha, beta, "worst scaled errors", worst)


@pytest.mark.parametrize("alpha,beta", [(0.0, 0.0), (-2.0, -4.0)])
def test_bf16_many_heads(alpha, beta):
    """64 query / 8 K/V heads (80 head tiles of the QKV projection, 8 query
    heads per K/V head); two layers, q/k/v bias, a ragged row tile."""
    w = small_bf16(n_layers=2, d=512, hq=64, hkv=8, F=1024, n_select=150, selection="isolated", alpha=alpha,
                   beta=beta)
    layers = wl.make_layer_weights(w, "cuda")
    rng = np.random.default_rng(13)
    local = rng.random((1, w.capacity)) < 0.5
    sink = rng.random((1, w.capacity)) < 0.2
    s = Setup(w, weights=layers, local=local, sink=sink)
    Ks0, Vs0 = f64(s.K), f64(s.V)
    emb = f64(s.embed)
    ids = s.ids.cpu().numpy()
    worst = run_and_compare(s, LazyWeights(layers), Ks0, Vs0, [emb[ids[0]]], TOL["bf16"])
    s.close()
    print("many-head worst", worst)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_qk_norm_model_against_oracle(dtype):
    """Q/K normalisation (Budgeted KV-Cache Repair, Sec. 13.2; the Qwen3
    block): every Q and K head RMS-normalised with its own weights before
    RoPE, no q/k/v bias; bf16 (head_dim 128) and fp32 (head_dim 64)."""
    if dtype == "bf16":
        w = small_bf16(n_layers=2, qkv_bias=False, qk_norm=True, selection="isolated", alpha=-1.0, beta=-2.0)
    else:
        m = wl.ModelShape(1, 256, 4, 2, 64, 512, 10000.0, 1e-5, "f32", False, vocab=500, qk_norm=True)
        w = wl.Workload("f32_qknorm", 8, m, 1, 700, 640, 200, 40, alpha=-1.0, beta=-2.0, selection="units")
    layers = wl.make_layer_weights(w, "cuda")
    rng = np.random.default_rng(17)
    local = rng.random((1, w.capacity)) < 0.5
    sink = rng.random((1, w.capacity)) < 0.2
    s = Setup(w, weights=layers, local=local, sink=sink)
    Ks0, Vs0 = f64(s.K), f64(s.V)
    emb = f64(s.embed)
    ids = s.ids.cpu().numpy()
    worst = run_and_compare(s, LazyWeights(layers), Ks0, Vs0, [emb[ids[0]]], TOL[dtype])
    s.close()
    print("qk-norm", dtype, "worst", worst)


def test_bf16_batch_of_sequences():
    """Independent sequences sharing weights (seq-major rows, per-sequence
    caches and plans)."""
    w = small_bf16(batch=3, selection="isolated", n_select=70, alpha=-1.0, beta=0.0)
    layers = wl.make_layer_weights(w, "cuda")
    s = Setup(w, weights=layers)
    Ks0, Vs0 = f64(s.K), f64(s.V)
    emb = f64(s.embed)
    ids = s.ids.cpu().numpy()
    worst = run_and_compare(s, LazyWeights(layers), Ks0, Vs0, [emb[ids[b]] for b in range(3)], TOL["bf16"])
    s.close()
    print("batch worst", worst)


def test_empty_selection_is_a_no_op():
    w = small_bf16(n_layers=1)
    s = Setup(w, positions=[np.array([], np.int32)])
    K_in = s.K.clone()
    s.select()
    s.refresh()
    s.sync()
    assert torch.equal(s.K, K_in)
    s.close()


def scaled_err(got, want):
    return np.abs(np.asarray(got) - np.asarray(want)) / np.maximum(1.0, np.abs(np.asarray(want)))


@pytest.mark.slow
def test_llama8b_full_size_against_oracle():
    """The Llama-3-8B-shaped workload at full size (32 layers, N = 7680,
    282 positions in units of 32-64), the launch configuration the benchmark
    times.

    Elementwise tolerance on the K/V rows of layer 0, whose inputs are the
    same embedding rows on both sides.  From layer 1 on, each side reads its
    own rounded layer outputs, and this random-weight stack amplifies any
    rounding difference (in the oracle itself, one bf16 ulp on 1 % of the
    layer-0 inputs is already 2.3e-2 at layer 1 and grows to a 1.9 scaled
    error after 32 layers).  So every layer's K/V rows and the final hidden
    rows are held to a budget: the GPU's distance to the exact (unrounded
    float64) recurrence may be at most twice the bf16 oracle's own distance to
    it, in RMS and in max (the 2x-native-error budget of the pages' FP32
    control, Budgeted KV-Cache Repair Sec. 13.5)."""
    w = wl.WORKLOADS["llama8b"]
    s = Setup(w)
    Ks0, Vs0 = f64(s.K[0]), f64(s.V[0])
    emb = s.embed
    ids = s.ids.cpu().numpy()
    U = oracle.sorted_positions(s.positions[0])
    X_src = np.zeros((w.capacity, w.model.d_model))
    X_src[U] = f64(emb[torch.from_numpy(ids[0][U].astype(np.int64)).cuda()])
    K_in, V_in = s.K.clone(), s.V.clone()
    spec = oracle_spec(w)
    # layer 0 alone first: the refreshed rows X^1 depend on the inputs only,
    # so they are held elementwise to the tolerance; this run rewrites only
    # layer 0's selected K/V rows, which the full refresh rewrites before
    # reading them, so it leaves the full run's results unchanged
    s.select()
    s.refresh(0, 1, flags=0)
    s.sync()
    X1 = oracle.refresh_packed(spec, LazyWeights(s.layers), Ks0[:1], Vs0[:1], s.local_mask[0], s.sink_mask[0], U,
                               X_src, n_layers=1)[0]
    assert_close_rows(f64(s.hidden[:len(U)]), X1, TOL["bf16"], "refreshed rows after layer 0")
    s.select()
    s.refresh()
    s.sync()
    exact = dataclasses.replace(spec, dtype="f64")
    W = LazyWeights(s.layers)
    Xb, Kb, Vb, lb, sb = oracle.refresh_packed(spec, W, Ks0, Vs0, s.local_mask[0], s.sink_mask[0], U, X_src)
    Xe, Ke, Ve, _, _ = oracle.refresh_packed(exact, W, Ks0, Vs0, s.local_mask[0], s.sink_mask[0], U, X_src)
    Ut = torch.from_numpy(U)
    report = []
    for l in range(w.model.n_layers):
        for name, G, B, E in (("K", s.K, Kb, Ke), ("V", s.V, Vb, Ve)):
            g = f64(G[0, l][:, Ut])
            b, e = B[l][:, U], E[l][:, U]
            if l == 0:
                assert_close(g, b, TOL["bf16"], f"{name} layer {l}")
            eg, eo = scaled_err(g, e), scaled_err(b, e)
            rg, ro = float(np.sqrt(np.mean(eg ** 2))), float(np.sqrt(np.mean(eo ** 2)))
            report.append((l, name, rg, ro, float(eg.max()), float(eo.max())))
            assert rg <= 2 * ro + 1e-4, f"{name} layer {l}: rms error {rg:.3e} vs oracle {ro:.3e}"
            assert eg.max() <= 2 * eo.max() + 1e-3, f"{name} layer {l}: max error {eg.max():.3e} vs {eo.max():.3e}"
    g = f64(s.hidden[:len(U)])
    eg, eo = scaled_err(g, Xe), scaled_err(Xb, Xe)
    rg, ro = float(np.sqrt(np.mean(eg ** 2))), float(np.sqrt(np.mean(eo ** 2)))
    print("hidden rms/max gpu", rg, eg.max(), "oracle", ro, eo.max())
    for r in report[::8]:
        print("layer %d %s rms gpu %.3e oracle %.3e max gpu %.3e oracle %.3e" % r)
    assert rg <= 2 * ro + 1e-4 and eg.max() <= 2 * eo.max() + 1e-3
    keep = torch.ones(w.capacity, dtype=torch.bool, device=s.K.device)
    keep[Ut.to(s.K.device)] = False
    assert torch.equal(s.K[0][:, :, keep], K_in[0][:, :, keep])
    assert torch.equal(s.V[0][:, :, keep], V_in[0][:, :, keep])
    local_after, sink_after = kvr.kvr_read_meta(s.handle, 1, s.words)
    np.testing.assert_array_equal(local_after[0], oracle.bitmask_words(lb)[:s.words])
    s.close()


@pytest.mark.slow
@pytest.mark.parametrize("n_select", [257, 289, 313, 320])
def test_llama8b_layer_with_paired_row_tiles(n_select):
    """One Llama-3-8B-shaped layer (N = 7680) whose selection the QKV and
    down projections split into two row tiles given to one CTA together (two
    products of N = BN per K step, two accumulator windows at both ends of
    tensor memory sharing their middle columns): 257 rows (tiles of 144, the
    second holding one row; windows of 288 sharing 64), 289 and 313 (tiles of
    160; windows of 320 sharing 128) and 320 (two full tiles of 160).  The
    refreshed rows, the layer's K/V rows and the untouched rows against the
    oracle, elementwise."""
    base = wl.WORKLOADS["llama8b"]
    w = dataclasses.replace(base, model=dataclasses.replace(base.model, n_layers=1), n_select=n_select)
    s = Setup(w)
    assert s.n_rows == n_select
    Ks0, Vs0 = f64(s.K[0]), f64(s.V[0])
    ids = s.ids.cpu().numpy()
    U = oracle.sorted_positions(s.positions[0])
    X_src = np.zeros((w.capacity, w.model.d_model))
    X_src[U] = f64(s.embed[torch.from_numpy(ids[0][U].astype(np.int64)).cuda()])
    K_in, V_in = s.K.clone(), s.V.clone()
    s.select()
    s.refresh()
    s.sync()
    X1, K1, V1, _, _ = oracle.refresh_packed(oracle_spec(w), LazyWeights(s.layers), Ks0, Vs0, s.local_mask[0],
                                             s.sink_mask[0], U, X_src)
    assert_close_rows(f64(s.hidden[:len(U)]), X1, TOL["bf16"], "refreshed rows")
    Ut = torch.from_numpy(U)
    assert_close(f64(s.K[0, 0][:, Ut]), K1[0][:, U], TOL["bf16"], "K layer 0")
    assert_close(f64(s.V[0, 0][:, Ut]), V1[0][:, U], TOL["bf16"], "V layer 0")
    keep = torch.ones(w.capacity, dtype=torch.bool, device=s.K.device)
    keep[Ut.to(s.K.device)] = False
    assert torch.equal(s.K[0][:, :, keep], K_in[0][:, :, keep])
    assert torch.equal(s.V[0][:, :, keep], V_in[0][:, :, keep])
    s.close()


@pytest.mark.parametrize("sink_static", [False, True])
def test_bf16_seven_query_heads_per_kv_head_block_seams(sink_static):
    """The block-seam geometry at the Qwen2.5-7B head grouping: 7 query heads
    per K/V head (14 / 2 heads x 128, so a query tile holds 18 positions x 7
    heads = 126 MMA rows), q/k/v bias, alpha = -2, beta = -4; N = 2112 as 8
    independently prefilled blocks of 264 with seam windows tau = 64 under the
    asymmetric rule (896 rows, 8 intervals); blocks 2..8 local and their first
    4 positions the sinks S' ("kv-cross-attention-reuse", Sec. 6.3-6.4).  With
    a static sink set the beta penalty also reaches the refreshed S'."""
    base = wl.WORKLOADS["qwen7b_seam"]
    m = dataclasses.replace(base.model, n_layers=2, d_model=1792, n_q_heads=14, n_kv_heads=2, ffn_dim=1024,
                            vocab=1000)
    w = dataclasses.replace(base, name="seam_g7", model=m, capacity=2112, n_tokens=2112)
    layers = wl.make_layer_weights(w, "cuda")
    s = Setup(w, weights=layers, flags=kvr.KVR_SINK_STATIC if sink_static else 0)
    assert len(s.positions[0]) == 896
    Ks0, Vs0 = f64(s.K), f64(s.V)
    emb = f64(s.embed)
    ids = s.ids.cpu().numpy()
    worst = run_and_compare(s, LazyWeights(layers), Ks0, Vs0, [emb[ids[0]]], TOL["bf16"], sink_static=sink_static)
    s.close()
    print("7 heads per K/V head, sink_static", sink_static, "worst", worst)
