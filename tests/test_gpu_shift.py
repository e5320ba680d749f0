"""GPU parity of Shift and splice (kvr_shift, kvr_splice) against the oracle.

Shift ("Budgeted KV-Cache Repair for Evolving Contexts", Sec. 7.1, Eq. 2)
deletes a span and moves the rest of the cache down, rotating each moved key
by -d positions.  Splice ("Models Take Notes at Prefill: KV Cache Can Be
Editable and Composable", Sec. 5) places a block computed on its own at new
positions, rotating its keys by the position change.  Values and every
untouched row are compared bit for bit, the metadata words bit for bit, and
the rotated keys within one bf16 rounding of the float64 oracle (the kernel
rotates in fp32 with the angle formed in double, then rounds once)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from selective_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup  # noqa: E402
from helpers import TOL, assert_close, f64, small_bf16  # noqa: E402


def rotated_close(got, want, dtype):
    """One storage rounding of the exact value, plus fp32 arithmetic noise on
    the row's scale."""
    got, want = f64(got), np.asarray(want, dtype=np.float64)
    scale = np.max(np.abs(want), axis=-1, keepdims=True)
    rel = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -22
    bound = rel * np.abs(want) + 2.0 ** -20 * scale
    bad = np.abs(got - want) > bound
    assert not bad.any(), f"{bad.sum()} keys off by more than one rounding; worst {np.max(np.abs(got - want))}"


def fp32_model(dh):
    m = wl.ModelShape(2, 256, 4, 2, dh, 512, 10000.0, 1e-5, "f32", False, vocab=100)
    return wl.Workload(f"f32_dh{dh}", 8, m, 2, 700, 640, 200, 32)


def masks(w, n_tokens, seed):
    rng = np.random.default_rng(seed)
    local = rng.random((w.batch, w.capacity)) < 0.5
    sink = rng.random((w.batch, w.capacity)) < 0.1
    local[:, n_tokens:] = False
    sink[:, n_tokens:] = False
    return local, sink


def new_cache(w, n_tokens, suffix_start, local, sink):
    K, V = wl.make_random_cache(w, "cuda")
    h = kvr.kvr_create_cache(kvr.model_desc(w.model), w.batch, w.capacity, K, V, n_tokens, suffix_start,
                             np.ascontiguousarray(wl.pack_bits(local)), np.ascontiguousarray(wl.pack_bits(sink)))
    return h, K, V


SHIFT_CASES = [
    (300, 37),     # overlapping move, d smaller than a tile
    (0, 5),        # deletion at the very start
    (1000, 100),   # deletion at the end: nothing moves, the cache only shrinks
    (50, 700),     # d larger than the moved run: source and destination apart
    (301, 331),    # unaligned start and d (metadata words straddle)
]


@pytest.mark.parametrize("start,d", SHIFT_CASES)
def test_shift_bf16_matches_oracle(start, d):
    w = small_bf16(n_layers=3, batch=2, capacity=1200, n_tokens=1100, suffix_start=400)
    m = w.model
    n = w.n_tokens
    local, sink = masks(w, n, 5 + start)
    h, K, V = new_cache(w, n, w.suffix_start, local, sink)
    K0, V0 = K.clone(), V.clone()
    kvr.kvr_shift(h, start, d)
    kvr.kvr_sync_status(h)
    n_new = n - d
    assert kvr.kvr_cache_info(h) == (n_new, min(w.suffix_start, start))
    Kw, Vw = oracle.shift(f64(K0[..., :n, :]), f64(V0[..., :n, :]), start, d, m.rope_theta)
    assert torch.equal(K[..., :start, :], K0[..., :start, :])
    np.testing.assert_array_equal(f64(V[..., :n_new, :]), Vw)
    rotated_close(K[..., start:n_new, :], Kw[..., start:, :], "bf16")
    # rows past the new end keep what they held
    assert torch.equal(K[..., n_new:, :], K0[..., n_new:, :])
    assert torch.equal(V[..., n_new:, :], V0[..., n_new:, :])
    lw, sw = kvr.kvr_read_meta(h, w.batch, (w.capacity + 31) // 32)
    for b in range(w.batch):
        np.testing.assert_array_equal(lw[b], oracle.bitmask_words(oracle.shift_mask(local[b], start, d)))
        np.testing.assert_array_equal(sw[b], oracle.bitmask_words(oracle.shift_mask(sink[b], start, d)))
    kvr.kvr_destroy_cache(h)


@pytest.mark.parametrize("dh", [64, 128])
def test_shift_fp32_matches_oracle(dh):
    w = fp32_model(dh)
    n, start, d = w.n_tokens, 211, 45
    local, sink = masks(w, n, 9)
    h, K, V = new_cache(w, n, w.suffix_start, local, sink)
    K0, V0 = K.clone(), V.clone()
    kvr.kvr_shift(h, start, d)
    kvr.kvr_sync_status(h)
    Kw, Vw = oracle.shift(f64(K0[..., :n, :]), f64(V0[..., :n, :]), start, d, w.model.rope_theta)
    np.testing.assert_array_equal(f64(V[..., :n - d, :]), Vw)
    assert torch.equal(K[..., :start, :], K0[..., :start, :])
    rotated_close(K[..., start:n - d, :], Kw[..., start:, :], "f32")
    kvr.kvr_destroy_cache(h)


def test_shift_validation_and_state():
    w = small_bf16(n_layers=1, capacity=600, n_tokens=560, suffix_start=100, n_select=20)
    s = Setup(w)
    K0 = s.K.clone()
    for start, d in [(-1, 3), (0, -1), (550, 11), (0, 560)]:
        with pytest.raises(kvr.KvrError) as e:
            kvr.kvr_shift(s.handle, start, d)
        assert e.value.status == kvr.KVR_EINVAL
    kvr.kvr_shift(s.handle, 200, 0)                       # d = 0: nothing
    kvr.kvr_sync_status(s.handle)
    assert torch.equal(s.K, K0)
    assert kvr.kvr_cache_info(s.handle) == (560, 100)
    s.select()
    kvr.kvr_shift(s.handle, 60, 10)                       # deletion inside the prefix
    assert kvr.kvr_cache_info(s.handle) == (550, 60)
    with pytest.raises(kvr.KvrError) as e:                # the selection was dropped
        s.refresh()
    assert e.value.status == kvr.KVR_ESTATE
    with pytest.raises(kvr.KvrError) as e:                # position 555 is past the new end
        kvr.kvr_select(s.handle, np.array([555], np.int32), np.array([1], np.int32), -1, token_ids=s.ids,
                       embed_table=s.embed, vocab=w.model.vocab, hidden_out=s.hidden)
    assert e.value.status == kvr.KVR_ERANGE
    s.positions = [np.arange(300, 320)]
    s.pos_host = np.ascontiguousarray(s.positions[0].astype(np.int32))
    s.counts = np.array([20], np.int32)
    assert s.select() == (20, 1)
    s.refresh()
    s.sync()
    s.close()


def test_shift_then_refresh_matches_oracle_edit_flow():
    """The whole edit on the tiny fp32 model: the stale cache is the oracle's
    prefill of the pre-edit sequence (1100 tokens); Shift deletes [256, 332)
    on the GPU; the refresh then recomputes 64 positions of the retained
    suffix from the edited sequence's inputs.  The oracle runs the same edit
    (shift, then the packed refresh) in float64."""
    base = wl.WORKLOADS["tiny"]
    start, d = 256, 76
    w0 = dataclasses.replace(base, capacity=1100, n_tokens=1100, suffix_start=start)
    spec = oracle.Spec.of(base.model)
    lc = wl.make_layer_weights(base, "cpu")
    W = [{k: f64(v) if v is not None else None for k, v in L.items()} for L in lc]
    X_orig = f64(wl.make_hidden_inputs(w0, "cpu"))[0]
    _, Ks, Vs = oracle.prefill(spec, W, X_orig)
    X_edit = np.concatenate([X_orig[:start], X_orig[start + d:]])
    positions = wl.make_positions(base)
    s = Setup(w0, cache=(torch.from_numpy(Ks[None]).float().cuda(), torch.from_numpy(Vs[None]).float().cuda()),
              weights=[{k: v.cuda() if v is not None else None for k, v in L.items()} for L in lc],
              positions=positions)
    src = torch.zeros((1, w0.capacity, base.model.d_model), dtype=torch.float32)
    src[0, :len(X_edit)] = torch.from_numpy(X_edit)
    s.hidden_src = src.cuda()
    kvr.kvr_shift(s.handle, start, d)
    assert kvr.kvr_cache_info(s.handle) == (1024, start)
    s.select()
    s.refresh()
    s.sync()
    K0, V0 = oracle.shift(Ks, Vs, start, d, spec.rope_theta)
    X, K, V, _, _ = oracle.refresh_packed(spec, W, K0, V0, np.zeros(1024, bool), np.zeros(1024, bool),
                                          positions[0], X_edit)
    U = oracle.sorted_positions(positions[0])
    assert_close(f64(s.hidden[:len(U)]), X, TOL["f32"], "hidden rows")
    assert_close(f64(s.K[0][..., :1024, :]), K, TOL["f32"], "K after shift and refresh")
    assert_close(f64(s.V[0][..., :1024, :]), V, TOL["f32"], "V after shift and refresh")
    s.close()


@pytest.mark.parametrize("src_pos,dst_pos,flags", [(0, 700, kvr.KVR_SPLICE_LOCAL | kvr.KVR_SPLICE_SINK),
                                                   (37, 37, 0), (900, 5, kvr.KVR_SPLICE_LOCAL)])
def test_splice_matches_oracle(src_pos, dst_pos, flags):
    w = small_bf16(n_layers=2, batch=2, capacity=1200, n_tokens=1100, suffix_start=0)
    m = w.model
    n_blk = 300
    local, sink = masks(w, w.n_tokens, 13)
    h, K, V = new_cache(w, w.n_tokens, 0, local, sink)
    K0, V0 = K.clone(), V.clone()
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    shape = (m.n_layers, m.n_kv_heads, n_blk, m.head_dim)
    kb = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    vb = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    seq = 1
    kvr.kvr_splice(h, seq, dst_pos, n_blk, kb, vb, src_pos, flags)
    kvr.kvr_sync_status(h)
    Kw, Vw = oracle.reposition(f64(kb), f64(vb), src_pos, dst_pos, m.rope_theta)
    rows = slice(dst_pos, dst_pos + n_blk)
    if src_pos == dst_pos:
        assert torch.equal(K[seq][..., rows, :], kb)          # a rotation by zero is exact
    rotated_close(K[seq][..., rows, :], Kw, "bf16")
    np.testing.assert_array_equal(f64(V[seq][..., rows, :]), Vw)
    keep = torch.ones(w.capacity, dtype=torch.bool, device="cuda")
    keep[rows] = False
    assert torch.equal(K[seq][..., keep, :], K0[seq][..., keep, :])
    assert torch.equal(V[seq][..., keep, :], V0[seq][..., keep, :])
    assert torch.equal(K[0], K0[0]) and torch.equal(V[0], V0[0])
    lw, sw = kvr.kvr_read_meta(h, w.batch, (w.capacity + 31) // 32)
    want_l, want_s = local.copy(), sink.copy()
    if flags & kvr.KVR_SPLICE_LOCAL:
        want_l[seq, rows] = True
    if flags & kvr.KVR_SPLICE_SINK:
        want_s[seq, dst_pos:dst_pos + 4] = True
    for b in range(w.batch):
        np.testing.assert_array_equal(lw[b], oracle.bitmask_words(want_l[b]))
        np.testing.assert_array_equal(sw[b], oracle.bitmask_words(want_s[b]))
    for args in [(2, 0, 10), (0, 1095, 10), (0, -1, 10), (-1, 0, 10)]:
        with pytest.raises(kvr.KvrError):
            kvr.kvr_splice(h, *args, kb, vb, 0, 0)
    kvr.kvr_destroy_cache(h)


@pytest.mark.slow
def test_shift_full_size_llama_edit():
    """The Llama-3-8B-shaped edit at full size: an 8192-token cache (32
    layers, 8 K/V heads) loses the 512-token span at 2048.  Every value row
    and every untouched key row is compared bit for bit; the moved keys of
    sampled (layer, head) slabs against the oracle."""
    w = dataclasses.replace(wl.WORKLOADS["llama8b"], n_tokens=8192)
    local, sink = masks(w, 8192, 21)
    h, K, V = new_cache(w, 8192, 2048, local, sink)
    K0, V0 = K.clone(), V.clone()
    kvr.kvr_shift(h, 2048, 512)
    kvr.kvr_sync_status(h)
    assert kvr.kvr_cache_info(h) == (7680, 2048)
    assert torch.equal(V[..., :7680, :], torch.cat([V0[..., :2048, :], V0[..., 2560:, :]], dim=-2))
    assert torch.equal(K[..., :2048, :], K0[..., :2048, :])
    assert torch.equal(K[..., 7680:, :], K0[..., 7680:, :])
    for layer, head in [(0, 0), (17, 3), (31, 7)]:
        Kw, _ = oracle.shift(f64(K0[0, layer, head]), f64(V0[0, layer, head]), 2048, 512, w.model.rope_theta)
        rotated_close(K[0, layer, head, 2048:7680], Kw[2048:], "bf16")
    lw, sw = kvr.kvr_read_meta(h, 1, 256)
    np.testing.assert_array_equal(lw[0], oracle.bitmask_words(oracle.shift_mask(local[0], 2048, 512)))
    np.testing.assert_array_equal(sw[0], oracle.bitmask_words(oracle.shift_mask(sink[0], 2048, 512)))
    kvr.kvr_destroy_cache(h)
