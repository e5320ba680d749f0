"""An independent pin of the oracle's decoder block (CPU only).

The closed forms in test_oracle_refresh.py (whole-suffix refresh = prefill,
packed = interval-wise) tie the oracle's schedules to each other, but the
packed-row layer and the prefill share their primitives, so a mistake inside
the block (the SwiGLU activation, which half of the gate/up projection is
gated, where the residuals and the second RMSNorm sit, the LoRA or Q/K-norm
placement) would show on both sides.  Here the block is written a second
time from torch.nn.functional in float64 -- F.rms_norm, F.linear, F.silu,
F.scaled_dot_product_attention with an additive causal + bias mask and
grouped-query heads, the rotary map as a complex multiplication -- and the
oracle (float64, no storage rounding) must agree with it to 1e-12.

The block follows "Budgeted KV-Cache Repair for Evolving Contexts",
Sec. 13.2 (the recompute runs the model's own projections, Q/K
normalisation, rotary map, attention, residuals, normalisation and MLP;
Eq. 21 writes the fresh K/V rows before the attention of the layer, Eq. 22
attends over the whole cache up to and including the row's own position)
and the logit bias of "kv-cross-attention-reuse", Sec. 6.4.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import Spec

TOL = 1e-12


def rope_complex(x, pos, theta):
    """Rotary map as a complex multiplication: dimension pairs (i, i + d/2)
    form z = x_i + j x_{i+d/2}, multiplied by exp(j pos theta^(-2i/d)).
    x [..., n, d], pos [n]."""
    d = x.shape[-1]
    half = d // 2
    inv = torch.pow(torch.tensor(float(theta), dtype=torch.float64),
                    -2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = pos.to(torch.float64)[:, None] * inv[None, :]
    z = torch.complex(x[..., :half], x[..., half:]) * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([z.real, z.imag], dim=-1)


def torch_block(spec, W, X, K, V, pos, bias, allowed=None):
    """One pre-norm decoder layer for rows X [R, d] at positions pos [R] over
    the caches K, V [H_kv, N, d_h] (the rows at pos are overwritten first).
    Returns (X_next, K, V).  allowed [R, N] (optional) restricts the keys
    further (independently prefilled blocks)."""
    Hq, Hkv, dh, Fd, eps = spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.ffn_dim, spec.rms_eps
    R, d = X.shape
    N = K.shape[1]
    t = lambda a: None if a is None else torch.as_tensor(a, dtype=torch.float64)
    X = t(X)
    K, V = t(K).clone(), t(V).clone()
    pos = torch.as_tensor(np.asarray(pos), dtype=torch.int64)
    xn = F.rms_norm(X, (d,), weight=t(W["norm1"]), eps=eps)
    qkv = F.linear(xn, t(W["w_qkv"]), t(W.get("b_qkv")))
    q, k, v = qkv.split([Hq * dh, Hkv * dh, Hkv * dh], dim=-1)
    if W.get("a_q") is not None:
        q = q + F.linear(F.linear(xn, t(W["a_q"])), t(W["b_q"]))
        v = v + F.linear(F.linear(xn, t(W["a_v"])), t(W["b_v"]))
    q = q.reshape(R, Hq, dh)
    k = k.reshape(R, Hkv, dh)
    if W.get("q_norm") is not None:
        q = F.rms_norm(q, (dh,), weight=t(W["q_norm"]), eps=eps)
        k = F.rms_norm(k, (dh,), weight=t(W["k_norm"]), eps=eps)
    q = rope_complex(q.transpose(0, 1), pos, spec.rope_theta)       # [Hq, R, dh]
    k = rope_complex(k.transpose(0, 1), pos, spec.rope_theta)       # [Hkv, R, dh]
    K[:, pos] = k
    V[:, pos] = v.reshape(R, Hkv, dh).transpose(0, 1)
    keep = torch.arange(N)[None, :] <= pos[:, None]
    if allowed is not None:
        keep = keep & torch.as_tensor(allowed)
    mask = torch.where(keep, t(bias)[None, :].expand(R, N), torch.tensor(-math.inf, dtype=torch.float64))
    o = F.scaled_dot_product_attention(q[None], K[None], V[None], attn_mask=mask, scale=1.0 / math.sqrt(dh),
                                       enable_gqa=True)[0]          # [Hq, R, dh]
    h = X + F.linear(o.transpose(0, 1).reshape(R, Hq * dh), t(W["w_o"]))
    hn = F.rms_norm(h, (d,), weight=t(W["norm2"]), eps=eps)
    gate, up = F.linear(hn, t(W["w_gate_up"])).split([Fd, Fd], dim=-1)
    return h + F.linear(F.silu(gate) * up, t(W["w_down"])), K, V


def make_case(seed, *, hq=4, hkv=2, dh=16, d=48, Fd=40, N=40, bias=False, lora=False, qk_norm=False):
    rng = np.random.default_rng(seed)
    spec = Spec(1, d, hq, hkv, dh, Fd, 10000.0, 1e-5, "f64")
    qkv = (hq + 2 * hkv) * dh
    W = {
        "w_qkv": rng.standard_normal((qkv, d)) * 0.2,
        "b_qkv": rng.standard_normal(qkv) * 0.2 if bias else None,
        "w_o": rng.standard_normal((d, hq * dh)) * 0.2,
        "w_gate_up": rng.standard_normal((2 * Fd, d)) * 0.2,
        "w_down": rng.standard_normal((d, Fd)) * 0.2,
        "norm1": 1.0 + 0.1 * rng.standard_normal(d),
        "norm2": 1.0 + 0.1 * rng.standard_normal(d),
    }
    if lora:
        r = 3
        W.update(a_q=rng.standard_normal((r, d)) * 0.3, b_q=rng.standard_normal((hq * dh, r)) * 0.3,
                 a_v=rng.standard_normal((r, d)) * 0.3, b_v=rng.standard_normal((hkv * dh, r)) * 0.3)
    if qk_norm:
        W.update(q_norm=1.0 + 0.1 * rng.standard_normal(dh), k_norm=1.0 + 0.1 * rng.standard_normal(dh))
    K = rng.standard_normal((hkv, N, dh))
    V = rng.standard_normal((hkv, N, dh))
    return rng, spec, W, K, V


@pytest.mark.parametrize("bias,lora,qk_norm,alpha,beta", [
    (False, False, False, 0.0, 0.0),
    (True, False, False, -2.0, -4.0),
    (False, True, False, 1.0, -3.0),
    (True, False, True, -1.5, 0.5),
    (True, True, True, 2.0, -2.0),
])
def test_layer_rows_matches_torch_functional_block(bias, lora, qk_norm, alpha, beta):
    rng, spec, W, K, V = make_case(3, bias=bias, lora=lora, qk_norm=qk_norm)
    N = K.shape[1]
    pos = np.sort(rng.choice(np.arange(5, N), size=9, replace=False))
    X = rng.standard_normal((len(pos), spec.d_model))
    local = rng.random(N) < 0.5
    sink = rng.random(N) < 0.3
    b = alpha * local + beta * sink
    Ko, Vo = K.copy(), V.copy()
    got = oracle.layer_rows(spec, W, X, Ko, Vo, pos, b)
    want, Kt, Vt = torch_block(spec, W, X, K, V, pos, b)
    np.testing.assert_allclose(got, want.numpy(), rtol=0, atol=TOL * max(1.0, float(np.abs(got).max())))
    np.testing.assert_allclose(Ko, Kt.numpy(), rtol=0, atol=TOL)
    np.testing.assert_allclose(Vo, Vt.numpy(), rtol=0, atol=TOL)


@pytest.mark.parametrize("blocks,lora,qk_norm", [(False, False, False), (True, False, True), (False, True, False)])
def test_prefill_matches_torch_functional_block(blocks, lora, qk_norm):
    """Two layers of the whole-sequence prefill (optionally independently
    prefilled blocks at their global positions) against the torch block run
    over every position."""
    rng, spec, W0, _, _ = make_case(5, bias=True, lora=lora, qk_norm=qk_norm)
    _, _, W1, _, _ = make_case(6, bias=True, lora=lora, qk_norm=qk_norm)
    spec = Spec(2, spec.d_model, spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.ffn_dim, spec.rope_theta,
                spec.rms_eps, "f64")
    N = 30
    X = rng.standard_normal((N, spec.d_model))
    bounds = [(0, 12), (12, 30)] if blocks else None
    got_X, got_K, got_V = oracle.prefill(spec, [W0, W1], X, block_bounds=bounds)
    allowed = None
    if blocks:
        bid = np.zeros(N, int)
        bid[12:] = 1
        allowed = bid[:, None] == bid[None, :]
    pos = np.arange(N)
    x = X
    for l, W in enumerate((W0, W1)):
        K = np.zeros((spec.n_kv_heads, N, spec.head_dim))
        V = np.zeros_like(K)
        x, Kt, Vt = torch_block(spec, W, x, K, V, pos, np.zeros(N), allowed)
        x = x.numpy()
        np.testing.assert_allclose(got_K[l], Kt.numpy(), rtol=0, atol=TOL)
        np.testing.assert_allclose(got_V[l], Vt.numpy(), rtol=0, atol=TOL)
    np.testing.assert_allclose(got_X, x, rtol=0, atol=TOL * max(1.0, float(np.abs(x).max())))


def test_torch_block_detects_a_swapped_gate():
    """The comparison is sharp: gating the up half instead of the gate half
    (a plausible slip) moves the output far beyond the tolerance."""
    rng, spec, W, K, V = make_case(7)
    pos = np.array([10, 11, 30])
    X = rng.standard_normal((3, spec.d_model))
    want = torch_block(spec, W, X, K, V, pos, np.zeros(K.shape[1]))[0].numpy()
    Fd = spec.ffn_dim
    Wswap = dict(W, w_gate_up=np.concatenate([W["w_gate_up"][Fd:], W["w_gate_up"][:Fd]]))
    got = oracle.layer_rows(spec, Wswap, X, K.copy(), V.copy(), pos, np.zeros(K.shape[1]))
    assert np.abs(got - want).max() > 1e-3
