"""Pins for the oracle's arithmetic (CPU only).

Every function is pinned to something other than itself: brute-force loops
written with the standard library, library routines (torch's bf16 cast,
complex multiplication), closed forms the pages state (whole-suffix refresh
equals a prefill of the edited sequence; packed equals interval-wise;
degeneration of the biased operator), and invariants (unselected K/V rows
untouched, RoPE relativity).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import Spec

# ----------------------------------------------------------------------------
# storage rounding
# ----------------------------------------------------------------------------


def test_round_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 3.4e38], np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_round_bf16_ties_and_double_rounding():
    e = 2.0 ** -7   # bf16 quantum on [1, 2)
    assert oracle.round_bf16(1 + e / 2) == 1.0                 # tie -> even
    assert oracle.round_bf16(1 + 3 * e / 2) == 1 + 2 * e      # tie -> even (up)
    # direct rounding from float64: just above the tie goes up, although a
    # detour through float32 would land on the tie and then round down
    x = 1 + e / 2 + 2.0 ** -30
    assert np.float32(x) == np.float32(1 + e / 2)
    assert oracle.round_bf16(x) == 1 + e
    assert oracle.round_bf16(-x) == -(1 + e)
    assert np.isinf(oracle.round_bf16(3.5e38))
    # subnormals are multiples of 2^-133, ties to even
    assert oracle.round_bf16(2.0 ** -140) == 0.0
    assert oracle.round_bf16(2.0 ** -133) == 2.0 ** -133
    assert oracle.round_bf16(1.5 * 2.0 ** -133) == 2.0 ** -132
    assert oracle.round_bf16(2.5 * 2.0 ** -133) == 2.0 ** -132


# ----------------------------------------------------------------------------
# primitives
# ----------------------------------------------------------------------------


def test_rms_norm_closed_form():
    x = np.array([[3.0, 4.0]])
    w = np.array([2.0, 0.5])
    eps = 1e-5
    r = math.sqrt((9 + 16) / 2 + eps)
    np.testing.assert_allclose(oracle.rms_norm(x, w, eps), [[6 / r, 2 / r]], rtol=1e-15)


def test_rope_against_complex_rotation():
    rng = np.random.default_rng(1)
    dh, n, theta = 16, 9, 10000.0
    x = rng.standard_normal((3, n, dh))
    pos = rng.integers(-500, 5000, size=n)
    got = oracle.rope(x, pos, theta)
    half = dh // 2
    for i in range(half):
        freq = theta ** (-(2 * i) / dh)
        z = (x[..., i] + 1j * x[..., i + half]) * np.exp(1j * pos * freq)
        np.testing.assert_allclose(got[..., i], z.real, atol=1e-12)
        np.testing.assert_allclose(got[..., i + half], z.imag, atol=1e-12)


def test_rope_group_properties():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 5, 128))
    a = rng.integers(0, 9000, 5)
    d = 512
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(5), 5e5), x)
    np.testing.assert_allclose(np.linalg.norm(oracle.rope(x, a, 5e5), axis=-1),
                               np.linalg.norm(x, axis=-1), rtol=1e-12)
    # Eq. 2 identity: R_{i-d} R_i^{-1} R_i x = R_{i-d} x
    np.testing.assert_allclose(oracle.rope(oracle.rope(x, a, 5e5), np.full(5, -d), 5e5),
                               oracle.rope(x, a - d, 5e5), atol=1e-9)


def _attention_brute(q, K, V, g, bias):
    """Per-element loops with math.exp; K/V heads expanded the way a
    grouped-query model repeats them (np.repeat along the head axis)."""
    R, Hq, dh = q.shape
    G = Hq // K.shape[0]
    Kr = np.repeat(K, G, axis=0)
    Vr = np.repeat(V, G, axis=0)
    out = np.zeros_like(q)
    for i in range(R):
        for h in range(Hq):
            s = [sum(q[i, h, t] * Kr[h, j, t] for t in range(dh)) / math.sqrt(dh) + bias[j]
                 for j in range(int(g[i]) + 1)]
            m = max(s)
            e = [math.exp(v - m) for v in s]
            z = sum(e)
            for t in range(dh):
                out[i, h, t] = sum(e[j] * Vr[h, j, t] for j in range(len(e))) / z
    return out


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 2), (6, 2), (4, 4)])
def test_attention_brute_force(Hq, Hkv):
    rng = np.random.default_rng(10 + Hq * 7 + Hkv)
    N, dh, R = 23, 8, 7
    q = rng.standard_normal((R, Hq, dh))
    K = rng.standard_normal((Hkv, N, dh))
    V = rng.standard_normal((Hkv, N, dh))
    g = np.sort(rng.choice(N, size=R, replace=False))
    loc = rng.random(N) < 0.4
    snk = rng.random(N) < 0.2
    for alpha, beta in [(0.0, 0.0), (-2.0, -4.0), (1.0, 0.0), (0.0, -4.0)]:
        bias = alpha * loc + beta * snk
        np.testing.assert_allclose(oracle.attention(q, K, V, g, bias),
                                   _attention_brute(q, K, V, g, bias), atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(5)
    N, dh = 40, 16
    q = rng.standard_normal((3, 2, dh))
    V = rng.standard_normal((1, N, dh))
    K = np.repeat(rng.standard_normal((1, 1, dh)), N, axis=1)  # all keys equal
    g = np.array([0, 10, 39])
    out = oracle.attention(q, K, V, g)
    for i, gi in enumerate(g):   # uniform weights over the visible prefix
        np.testing.assert_allclose(out[i, 0], V[0, :gi + 1].mean(axis=0), atol=1e-12)
    # a dominant bias selects one key
    bias = np.zeros(N)
    bias[7] = 1000.0
    K2 = rng.standard_normal((1, N, dh))
    out = oracle.attention(q, K2, V, np.array([20, 20, 20]), bias)
    np.testing.assert_allclose(out[:, 0], np.repeat(V[0, 7][None], 3, axis=0), atol=1e-12)
    # adding the same constant to every logit changes nothing
    b = rng.standard_normal(N)
    np.testing.assert_allclose(oracle.attention(q, K2, V, g, b), oracle.attention(q, K2, V, g, b + 3.0),
                               atol=1e-12)


def test_degeneration_empty_masks():
    """F equals Softmax(QK^T/sqrt d)V when the correction masks are empty or
    alpha = beta = 0 (kv-cross-attention-reuse, Sec. 6.4, Degeneration)."""
    rng = np.random.default_rng(6)
    q = rng.standard_normal((5, 4, 8))
    K = rng.standard_normal((2, 30, 8))
    V = rng.standard_normal((2, 30, 8))
    pos = np.array([3, 9, 10, 20, 29])
    loc = rng.random(30) < 0.5
    snk = rng.random(30) < 0.5
    plain = oracle.attention(q, K, V, pos)
    np.testing.assert_allclose(oracle.attend(q, K, V, pos, loc, snk, 0.0, 0.0), plain, atol=1e-14)
    np.testing.assert_allclose(oracle.attend(q, K, V, pos, np.zeros(30), np.zeros(30), -2.0, -4.0),
                               plain, atol=1e-14)
    assert not np.allclose(oracle.attend(q, K, V, pos, loc, snk, -2.0, -4.0), plain)


def test_lora_unmerged_equals_merged():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 12))
    W = rng.standard_normal((9, 12))
    A = rng.standard_normal((3, 12))
    Bm = rng.standard_normal((9, 3))
    np.testing.assert_allclose(x @ W.T + oracle.lora_delta(x, A, Bm), x @ (W + Bm @ A).T, atol=1e-12)


# ----------------------------------------------------------------------------
# the recurrence
# ----------------------------------------------------------------------------


def tiny_model(seed, L=2, d=32, Hq=4, Hkv=2, dh=8, F=48, bias=True, lora=False, dtype="f64"):
    rng = np.random.default_rng(seed)
    spec = Spec(L, d, Hq, Hkv, dh, F, 10000.0, 1e-5, dtype)
    W = []
    for _ in range(L):
        w = {
            "w_qkv": rng.standard_normal(((Hq + 2 * Hkv) * dh, d)) * 0.2,
            "b_qkv": rng.standard_normal((Hq + 2 * Hkv) * dh) * 0.2 if bias else None,
            "w_o": rng.standard_normal((d, Hq * dh)) * 0.2,
            "w_gate_up": rng.standard_normal((2 * F, d)) * 0.2,
            "w_down": rng.standard_normal((d, F)) * 0.2,
            "norm1": 1 + 0.1 * rng.standard_normal(d),
            "norm2": 1 + 0.1 * rng.standard_normal(d),
        }
        if lora:
            w.update(a_q=rng.standard_normal((2, d)) * 0.1, b_q=rng.standard_normal((Hq * dh, 2)) * 0.1,
                     a_v=rng.standard_normal((2, d)) * 0.1, b_v=rng.standard_normal((Hkv * dh, 2)) * 0.1)
        W.append(w)
    return spec, W


@pytest.mark.parametrize("lora", [False, True])
def test_whole_suffix_refresh_equals_prefill(lora):
    """Selecting the whole retained suffix recomputes it exactly: the result
    is a full prefill of the edited sequence (Budgeted KV-Cache Repair,
    Sec. 3.1 / 7.1: Replay retains the valid prefix and recomputes the
    suffix)."""
    spec, W = tiny_model(11, lora=lora)
    rng = np.random.default_rng(12)
    N, P = 40, 15
    clean = rng.standard_normal((N, spec.d_model))
    dirty = clean.copy()
    dirty[P:] += 0.7 * rng.standard_normal((N - P, spec.d_model))
    _, Ks, Vs = oracle.prefill(spec, W, dirty)          # stale cache
    Xp, Kp, Vp = oracle.prefill(spec, W, clean)         # fresh reference
    local = np.zeros(N, bool)
    local[P:] = True
    perm = rng.permutation(np.arange(P, N))
    X, K, V, loc2, _ = oracle.refresh_packed(spec, W, Ks, Vs, local, np.zeros(N, bool), perm, clean,
                                             alpha=-1.5, beta=0.0)
    np.testing.assert_allclose(X, Xp[P:], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(K, Kp, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(V, Vp, rtol=1e-11, atol=1e-11)
    assert not loc2.any()
    # the stale cache really was different
    assert np.abs(Ks[:, :, P:] - Kp[:, :, P:]).max() > 1e-2


def test_prefill_block_mask_is_relative_position_invariant():
    """Independently prefilled blocks at global positions (kv-cross-attention
    -reuse Sec. 6.1-6.2): each block's outputs equal a prefill of that block
    alone (RoPE depends only on relative position), and its keys are those
    keys rotated to the global offset."""
    spec, W = tiny_model(13, L=2)
    rng = np.random.default_rng(14)
    N, size = 36, 12
    X = rng.standard_normal((N, spec.d_model))
    bounds = [(i * size, (i + 1) * size) for i in range(3)]
    Xb, Kb, Vb = oracle.prefill(spec, W, X, block_bounds=bounds)
    for (s, e) in bounds:
        Xa, Ka, Va = oracle.prefill(spec, W, X[s:e])
        np.testing.assert_allclose(Xb[s:e], Xa, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(Vb[:, :, s:e], Va, rtol=1e-10, atol=1e-10)
        Krot = oracle.rope(Ka.reshape(-1, e - s, spec.head_dim), np.full(e - s, s), spec.rope_theta)
        np.testing.assert_allclose(Kb[:, :, s:e], Krot.reshape(Ka.shape), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("sink_static", [False, True])
def test_packed_equals_interval_wise(sink_static):
    """Layer-major packing preserves the interval-major recurrence in real
    arithmetic (Budgeted KV-Cache Repair, Sec. 13.2), with the alpha/beta
    correction terms active."""
    spec, W = tiny_model(21, L=3)
    rng = np.random.default_rng(22)
    N, P = 64, 10
    Ks = rng.standard_normal((spec.n_layers, spec.n_kv_heads, N, spec.head_dim))
    Vs = rng.standard_normal((spec.n_layers, spec.n_kv_heads, N, spec.head_dim))
    X_src = rng.standard_normal((N, spec.d_model))
    local = rng.random(N) < 0.6
    sink = rng.random(N) < 0.3
    U = np.concatenate([np.arange(12, 15), [20], np.arange(30, 37), [40, 42], np.arange(60, 64)])
    a = oracle.refresh_packed(spec, W, Ks, Vs, local, sink, rng.permutation(U), X_src, -2.0, -4.0,
                              sink_static)
    b = oracle.refresh_interval(spec, W, Ks, Vs, local, sink, U, X_src, -2.0, -4.0, sink_static)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_allclose(x, y, rtol=1e-11, atol=1e-11)
    np.testing.assert_array_equal(a[3], b[3])
    np.testing.assert_array_equal(a[4], b[4])


def test_packed_differs_from_commit_after_last_layer_reading():
    """Planted alternative: if selected keys kept their stale 'local' tilt
    until the end of the refresh, packed and interval-wise execution would
    disagree.  The oracle's reading (a selected key is fresh, hence global,
    whenever it is read) is the one under which they agree."""
    spec, W = tiny_model(23, L=2)
    rng = np.random.default_rng(24)
    N = 40
    Ks = rng.standard_normal((2, spec.n_kv_heads, N, spec.head_dim))
    Vs = rng.standard_normal((2, spec.n_kv_heads, N, spec.head_dim))
    X_src = rng.standard_normal((N, spec.d_model))
    local = np.ones(N, bool)
    U = np.array([5, 6, 7, 20, 21])
    b = oracle.refresh_interval(spec, W, Ks, Vs, local, np.zeros(N, bool), U, X_src, -2.0, 0.0)
    # planted: bias computed from the raw local bits (no selected-key exemption)
    K = Ks.copy()
    V = Vs.copy()
    X = X_src[U]
    for l in range(2):
        X = oracle.layer_rows(spec, W[l], X, K[l], V[l], U, -2.0 * local)
    assert np.abs(X - b[0]).max() > 1e-6


def test_unselected_rows_bit_identical():
    spec, W = tiny_model(31, L=2, dtype="bf16")
    rng = np.random.default_rng(32)
    N = 50
    Ks = oracle.round_bf16(rng.standard_normal((2, spec.n_kv_heads, N, spec.head_dim)))
    Vs = oracle.round_bf16(rng.standard_normal((2, spec.n_kv_heads, N, spec.head_dim)))
    U = np.array([30, 31, 45, 49])
    X, K, V, _, _ = oracle.refresh_packed(spec, W, Ks, Vs, np.ones(N, bool), np.zeros(N, bool), U,
                                          rng.standard_normal((N, spec.d_model)))
    keep = np.setdiff1d(np.arange(N), U)
    np.testing.assert_array_equal(K[:, :, keep], Ks[:, :, keep])
    np.testing.assert_array_equal(V[:, :, keep], Vs[:, :, keep])
    assert np.array_equal(K[:, :, U], oracle.round_bf16(K[:, :, U]))   # stored values are bf16
    assert np.array_equal(X, oracle.round_bf16(X))


def test_shift_eq2():
    """Shift (Budgeted KV-Cache Repair, Sec. 7.1 Eq. 2): keys prefilled at
    position i and shifted by d equal the same pre-rotation keys placed at
    i - d; values move unchanged; the prefix is untouched."""
    rng = np.random.default_rng(51)
    N, start, d, dh, theta = 40, 10, 7, 16, 5e5
    raw = rng.standard_normal((2, 3, N, dh))
    K = oracle.rope(raw.reshape(-1, N, dh), np.arange(N), theta).reshape(raw.shape)
    V = rng.standard_normal((2, 3, N, dh))
    Kn, Vn = oracle.shift(K, V, start, d, theta)
    assert Kn.shape[-2] == N - d
    np.testing.assert_array_equal(Kn[..., :start, :], K[..., :start, :])
    np.testing.assert_array_equal(Vn[..., start:, :], V[..., start + d:, :])
    want = oracle.rope(raw[..., start + d:, :].reshape(-1, N - start - d, dh),
                       np.arange(start, N - d), theta).reshape(Kn[..., start:, :].shape)
    np.testing.assert_allclose(Kn[..., start:, :], want, atol=1e-10)
    # a deletion that reaches the end moves nothing and only shortens the cache
    Kt, Vt = oracle.shift(K, V, N - d, d, theta)
    np.testing.assert_array_equal(Kt, K[..., :N - d, :])
    np.testing.assert_array_equal(Vt, V[..., :N - d, :])


def test_refresh_range_equals_layerwise_definition():
    """Adapter-drift recovery (CacheReforge, Bounded Recovery): with the
    range covering every layer, recomputing the whole suffix from the layer-0
    boundary is a whole-suffix refresh, i.e. a prefill of the suffix."""
    spec, W = tiny_model(61, L=3, lora=True)
    rng = np.random.default_rng(62)
    N, P = 30, 12
    X_all = rng.standard_normal((N, spec.d_model))
    dirty = X_all.copy()
    dirty[P:] *= 1.3
    _, Ks, Vs = oracle.prefill(spec, W, dirty)
    Xp, Kp, Vp = oracle.prefill(spec, W, X_all)
    U = np.array([14, 20, 27])
    X, K, V, _, _ = oracle.refresh_range(spec, W, Ks, Vs, np.zeros(N, bool), np.zeros(N, bool), U, X_all,
                                         X_all, P, N, 0, 3)
    np.testing.assert_allclose(X, Xp[U], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(K[:, :, P:], Kp[:, :, P:], rtol=1e-10, atol=1e-10)
    # a range in the middle: layers outside it touch only U
    X2, K2, V2, _, _ = oracle.refresh_range(spec, W, Ks, Vs, np.zeros(N, bool), np.zeros(N, bool), U,
                                            X_all, X_all * 0.9, P, N, 1, 2)
    others = np.setdiff1d(np.arange(P, N), U)
    np.testing.assert_array_equal(K2[0][:, others], Ks[0][:, others])
    np.testing.assert_array_equal(K2[2][:, others], Ks[2][:, others])
    assert np.abs(K2[1][:, others] - Ks[1][:, others]).max() > 1e-3


def test_reposition_notes_sec5():
    """Repositioning (Models Take Notes at Prefill, Sec. 5): a block whose keys
    were rotated at src.. and then moved to dst.. equals the same pre-rotation
    keys rotated at dst.. directly; values are untouched; moves compose, and a
    move by zero is the identity."""
    rng = np.random.default_rng(53)
    n, dh, theta = 9, 16, 1e4
    raw = rng.standard_normal((2, 3, n, dh))
    V = rng.standard_normal((2, 3, n, dh))
    at = lambda p0: oracle.rope(raw.reshape(-1, n, dh), np.arange(p0, p0 + n), theta).reshape(raw.shape)
    K5 = at(5)
    Kd, Vd = oracle.reposition(K5, V, 5, 1000, theta)
    np.testing.assert_allclose(Kd, at(1000), atol=1e-10)
    np.testing.assert_array_equal(Vd, V)
    K2, _ = oracle.reposition(*oracle.reposition(K5, V, 5, 40, theta), 40, 1000, theta)
    np.testing.assert_allclose(K2, Kd, atol=1e-10)
    np.testing.assert_allclose(oracle.reposition(K5, V, 7, 7, theta)[0], K5, atol=0)
    # moving down by d is what Shift does to the moved suffix
    K = at(0)
    Ks, _ = oracle.shift(K, V, 2, 3, theta)
    np.testing.assert_allclose(Ks[..., 2:, :], oracle.reposition(K[..., 5:, :], V[..., 5:, :], 5, 2, theta)[0],
                               atol=1e-12)


def test_qk_norm_invariants():
    """Q/K normalisation (Budgeted KV-Cache Repair, Sec. 13.2; the Qwen3
    block): (1) with unit weights every stored key head has norm sqrt(d_h)
    (the rotary map preserves norms); (2) scaling the Q and K rows of the
    projection (and their bias) by any c > 0 leaves the layer unchanged."""
    spec, W = tiny_model(81, L=1, bias=True)
    spec = dataclasses.replace(spec, rms_eps=1e-12)
    dh, Hq, Hkv = spec.head_dim, spec.n_q_heads, spec.n_kv_heads
    for w in W:
        w["q_norm"] = np.ones(dh)
        w["k_norm"] = np.ones(dh)
    rng = np.random.default_rng(82)
    N = 20
    X = rng.standard_normal((N, spec.d_model))
    K = np.zeros((Hkv, N, dh))
    V = np.zeros((Hkv, N, dh))
    pos = np.arange(N)
    out1 = oracle.layer_rows(spec, W[0], X, K, V, pos, None)
    np.testing.assert_allclose(np.linalg.norm(K, axis=-1), np.sqrt(dh), rtol=1e-9)
    # scale invariance, with non-unit weights
    W[0]["q_norm"] = 1 + 0.2 * rng.standard_normal(dh)
    W[0]["k_norm"] = 1 + 0.2 * rng.standard_normal(dh)
    K1, V1 = np.zeros((Hkv, N, dh)), np.zeros((Hkv, N, dh))
    ref = oracle.layer_rows(spec, W[0], X, K1, V1, pos, None)
    Ws = dict(W[0])
    qk = slice(0, (Hq + Hkv) * dh)
    Ws["w_qkv"] = W[0]["w_qkv"].copy()
    Ws["w_qkv"][qk] *= 7.5
    Ws["b_qkv"] = W[0]["b_qkv"].copy()
    Ws["b_qkv"][qk] *= 7.5
    K2, V2 = np.zeros((Hkv, N, dh)), np.zeros((Hkv, N, dh))
    out2 = oracle.layer_rows(spec, Ws, X, K2, V2, pos, None)
    np.testing.assert_allclose(out2, ref, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(K2, K1, rtol=1e-9, atol=1e-12)
    # without the per-head normalisation the same scaling changes the result
    Wn = {k: v for k, v in Ws.items() if k not in ("q_norm", "k_norm")}
    Wn0 = {k: v for k, v in W[0].items() if k not in ("q_norm", "k_norm")}
    a = oracle.layer_rows(spec, Wn, X, np.zeros((Hkv, N, dh)), np.zeros((Hkv, N, dh)), pos, None)
    b = oracle.layer_rows(spec, Wn0, X, np.zeros((Hkv, N, dh)), np.zeros((Hkv, N, dh)), pos, None)
    assert np.max(np.abs(a - b)) > 1e-3
    assert out1.shape == ref.shape
