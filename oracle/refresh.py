"""Oracle: the selective-refresh recurrence in plain float64 numpy.

Sources (cited by page title and section):
  [BKR]  "Budgeted KV-Cache Repair for Evolving Contexts"
  [KVX]  "kv-cross-attention-reuse" (mixed cache and operator F), Sec. 6
  [CRF]  "CacheReforge: Bounded Recovery for Stale KV Caches under Evolving
         Adapters"
  [NOTES] "Models Take Notes at Prefill: KV Cache Can Be Editable and
         Composable" (re-rotating a chunk's keys to new positions), Sec. 5

Model block (the pages run dense Llama/Qwen decoders): pre-norm RMSNorm,
Q/K/V projections (+bias for Qwen2.5 shapes; per-head RMSNorm of Q and K
for Qwen3 shapes), rotate-half RoPE at global positions, grouped-query softmax attention with scale 1/sqrt(d_h), output
projection + residual, RMSNorm, SwiGLU MLP + residual.

Storage rounding.  Arithmetic is float64 throughout.  A value is rounded to
the model's storage dtype (fp32 or bf16, round-to-nearest-even) exactly where
the refresh stores a tensor in that dtype: the normalised rows fed to a
projection, the rotated queries, the K/V rows written to the cache, the
attention output, the SwiGLU output and the hidden rows handed to the next
layer.  The post-attention residual h is kept unrounded.

Layouts: weights in nn.Linear layout [out, in]; cache per sequence
[L, H_kv, N, d_h]; hidden rows [R, d].
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

from .select import effective_masks, intervals, sorted_positions

__all__ = [
    "Spec", "round_bf16", "round_store", "rms_norm", "qk_norm", "rope", "silu",
    "attention", "layer_rows", "refresh_packed", "refresh_interval",
    "refresh_range", "prefill", "shift", "reposition", "attend", "lora_delta",
]

BF16_MAX = float.fromhex("0x1.fep127")


@dataclasses.dataclass(frozen=True)
class Spec:
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    rope_theta: float
    rms_eps: float
    dtype: str  # "f32" | "bf16" | "f64" (no rounding; used by closed-form pins)

    @staticmethod
    def of(shape) -> "Spec":
        return Spec(shape.n_layers, shape.d_model, shape.n_q_heads, shape.n_kv_heads,
                    shape.head_dim, shape.ffn_dim, float(shape.rope_theta),
                    float(shape.rms_eps), shape.dtype)


# ----------------------------------------------------------------------------
# primitives
# ----------------------------------------------------------------------------

def round_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even), directly
    from float64 (no intermediate fp32 rounding).  bf16 has an 8-bit
    significand and fp32's exponent range: normal numbers are k * 2^(e-8)
    with 128 <= k < 256, subnormals are multiples of 2^-133."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e = np.frexp(ax)
    q = np.maximum(e - 8, -133)
    r = np.rint(np.ldexp(ax, -q))
    y = np.ldexp(r, q)
    y = np.where(y > BF16_MAX, np.inf, y)
    y = np.where(np.isfinite(ax), y, ax)
    return np.copysign(y, x)


def round_store(x, dtype: str):
    """Storage rounding for the model dtype."""
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def rms_norm(x, w, eps):
    """RMSNorm: x / sqrt(mean(x^2) + eps) * w over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w


def qk_norm(W, q, k, eps):
    """Q/K normalisation ([BKR] Sec. 13.2, which recomputes the selected
    rows with the model's own projections, its Q/K normalisation and its
    rotary map; the Qwen3 block): every query and key head is RMS-normalised
    over its d_h dimensions with its own weight vector before the rotary map.  q [R, Hq, d_h], k [R, Hkv, d_h]; a layer
    without q_norm/k_norm weights passes both through."""
    if W.get("q_norm") is None:
        return q, k
    return rms_norm(q, W["q_norm"], eps), rms_norm(k, W["k_norm"], eps)


def rope(x, pos, theta):
    """Rotate-half rotary map at global positions.

    x [..., n, d_h] with pos [n]: dimension pairs (i, i + d_h/2) rotate by the
    angle pos * theta^(-2i/d_h), i = 0 .. d_h/2 - 1.  The angle is formed in
    float64."""
    x = np.asarray(x, dtype=np.float64)
    dh = x.shape[-1]
    half = dh // 2
    inv = np.power(float(theta), -2.0 * np.arange(half, dtype=np.float64) / dh)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def attention(q, K, V, g, bias=None, row_chunk=256):
    """Biased causal grouped-query attention over a whole cache.

    q [R, Hq, d_h]; K, V [H_kv, N, d_h]; g [R] query positions; bias [N].
    For query row i and head h (K/V head h // (Hq/H_kv)):
        s_ij = <q_i, k_j> / sqrt(d_h) + bias_j   for j <= g_i
        o_i  = sum_j softmax_j(s_ij) v_j
    ([KVX] Sec. 6.4 "Logit form" with bias_j = alpha*1[local_j] +
    beta*1[j in S']; [BKR] Sec. 13.2 Eq. 22: 0:u_r includes u_r.)
    Rows are independent; they are evaluated in chunks only to bound memory.
    """
    q = np.asarray(q, dtype=np.float64)
    R, Hq, dh = q.shape
    Hkv, N, _ = K.shape
    G = Hq // Hkv
    g = np.asarray(g, dtype=np.int64)
    b = np.zeros(N) if bias is None else np.asarray(bias, dtype=np.float64)
    j = np.arange(N)
    out = np.zeros((R, Hq, dh))
    scale = 1.0 / np.sqrt(dh)
    for r0 in range(0, R, row_chunk):
        r1 = min(R, r0 + row_chunk)
        n_use = int(g[r0:r1].max()) + 1
        visible = j[None, :n_use] <= g[r0:r1, None]
        for h in range(Hq):
            kv = h // G
            s = q[r0:r1, h, :] @ K[kv, :n_use].T * scale + b[None, :n_use]
            s = np.where(visible, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=1, keepdims=True)
            out[r0:r1, h, :] = p @ V[kv, :n_use]
    return out


def lora_delta(x, a, b):
    """Low-rank adapter term (x A^T) B^T for A [r, in], B [out, r]
    ([CRF] Implementation: a LoRA on the cache-producing projections)."""
    return (x @ a.T) @ b.T


# ----------------------------------------------------------------------------
# one layer over packed rows
# ----------------------------------------------------------------------------

def layer_rows(spec: Spec, W, X, K, V, pos, bias):
    """One decoder layer for the packed rows X [R, d] at positions pos [R].

    Writes the fresh K/V rows into K, V ([H_kv, N, d_h], modified in place)
    before any attention of this layer ([BKR] Sec. 13.2 Eq. 21), then attends
    every row over the whole cache with its causal limit ([BKR] Eq. 22;
    [KVX] Sec. 6.4), and finishes with the output projection, residual,
    RMSNorm and SwiGLU MLP.  Returns the next layer's rows (rounded)."""
    rnd = lambda a: round_store(a, spec.dtype)
    Hq, Hkv, dh = spec.n_q_heads, spec.n_kv_heads, spec.head_dim
    R = X.shape[0]
    pos = np.asarray(pos, dtype=np.int64)

    xn = rnd(rms_norm(X, W["norm1"], spec.rms_eps))
    qkv = xn @ W["w_qkv"].T
    if W.get("b_qkv") is not None:
        qkv = qkv + W["b_qkv"]
    q = qkv[:, : Hq * dh]
    k = qkv[:, Hq * dh: (Hq + Hkv) * dh]
    v = qkv[:, (Hq + Hkv) * dh:]
    if W.get("a_q") is not None:
        q = q + lora_delta(xn, W["a_q"], W["b_q"])
        v = v + lora_delta(xn, W["a_v"], W["b_v"])
    q, k = qk_norm(W, q.reshape(R, Hq, dh), k.reshape(R, Hkv, dh), spec.rms_eps)
    q = rnd(rope(q.transpose(1, 0, 2), pos, spec.rope_theta)).transpose(1, 0, 2)
    k = rnd(rope(k.transpose(1, 0, 2), pos, spec.rope_theta))
    v = rnd(v.reshape(R, Hkv, dh).transpose(1, 0, 2))
    K[:, pos, :] = k
    V[:, pos, :] = v

    o = rnd(attention(q, K, V, pos, bias)).reshape(R, Hq * dh)
    h = X + o @ W["w_o"].T
    hn = rnd(rms_norm(h, W["norm2"], spec.rms_eps))
    gu = hn @ W["w_gate_up"].T
    F = spec.ffn_dim
    act = rnd(silu(gu[:, :F]) * gu[:, F:])
    return rnd(h + act @ W["w_down"].T)


def _bias(local, sink, selected, alpha, beta, sink_static):
    loc, snk = effective_masks(local, sink, selected, sink_static)
    return alpha * loc.astype(np.float64) + beta * snk.astype(np.float64)


def _commit(local, sink, pos, sink_static):
    """type_t <- global for refreshed t ([KVX] Sec. 6.4, physical repair);
    refreshed positions leave S' unless the sink set is static."""
    local[pos] = False
    if not sink_static:
        sink[pos] = False


# ----------------------------------------------------------------------------
# schedules
# ----------------------------------------------------------------------------

def refresh_packed(spec: Spec, weights, K, V, local, sink, positions, X_src,
                   alpha=0.0, beta=0.0, sink_static=False, n_layers=None):
    """Layer-major packed refresh of one sequence ([BKR] Sec. 3.3, Sec. 13.2).

    K, V [L, H_kv, N, d_h]; local, sink bool [N]; positions: the selected
    positions (any order); X_src [N, d]: the per-position layer-0 inputs (the
    gathered embedding rows or given hidden rows).  Returns
    (X [B, d] in sorted-position order, K, V, local, sink); inputs are not
    modified."""
    K = np.array(K, dtype=np.float64)
    V = np.array(V, dtype=np.float64)
    local = np.array(local, dtype=bool)
    sink = np.array(sink, dtype=bool)
    U = sorted_positions(positions)
    sel = np.zeros(local.shape[0], dtype=bool)
    sel[U] = True
    bias = _bias(local, sink, sel, alpha, beta, sink_static)
    X = round_store(np.asarray(X_src, dtype=np.float64)[U], spec.dtype)
    L = spec.n_layers if n_layers is None else n_layers
    for l in range(L):
        X = layer_rows(spec, weights[l], X, K[l], V[l], U, bias)
    _commit(local, sink, U, sink_static)
    return X, K, V, local, sink


def refresh_interval(spec: Spec, weights, K, V, local, sink, positions, X_src,
                     alpha=0.0, beta=0.0, sink_static=False, n_layers=None):
    """Interval-wise (sequential maximal-interval) refresh ([BKR] Sec. 7.1):
    each maximal interval [a, b) is forwarded through every layer against the
    cache as left by the earlier intervals, and its rows replace [a, b) at
    every layer.  Same return convention as refresh_packed."""
    K = np.array(K, dtype=np.float64)
    V = np.array(V, dtype=np.float64)
    local = np.array(local, dtype=bool)
    sink = np.array(sink, dtype=bool)
    U = sorted_positions(positions)
    X_src = np.asarray(X_src, dtype=np.float64)
    L = spec.n_layers if n_layers is None else n_layers
    out = {}
    for a, b in intervals(U):
        pos = np.arange(a, b)
        sel = np.zeros(local.shape[0], dtype=bool)
        sel[pos] = True
        bias = _bias(local, sink, sel, alpha, beta, sink_static)
        X = round_store(X_src[pos], spec.dtype)
        for l in range(L):
            X = layer_rows(spec, weights[l], X, K[l], V[l], pos, bias)
        _commit(local, sink, pos, sink_static)
        for i, p in enumerate(pos):
            out[int(p)] = X[i]
    Xs = np.stack([out[int(u)] for u in U]) if len(U) else np.zeros((0, spec.d_model))
    return Xs, K, V, local, sink


def refresh_range(spec: Spec, weights, K, V, local, sink, positions, X_src,
                  boundary, suffix_start, n_tokens, r0, r1, alpha=0.0, beta=0.0):
    """Adapter-drift repair of one sequence ([CRF] "Executable restart"):
    layers [r0, r1) are recomputed over the whole affected suffix
    [suffix_start, n_tokens), every other layer refreshes only `positions`.

    boundary [N, d]: the stored hidden state entering layer r0 from the
    original prefill.  Rows of the suffix that are not selected enter layer r0
    from it; selected rows keep their refreshed state.  After layer r1-1 the
    selected rows continue alone."""
    K = np.array(K, dtype=np.float64)
    V = np.array(V, dtype=np.float64)
    local = np.array(local, dtype=bool)
    sink = np.array(sink, dtype=bool)
    U = sorted_positions(positions)
    full = np.arange(suffix_start, n_tokens)
    X = round_store(np.asarray(X_src, dtype=np.float64)[U], spec.dtype)
    selU = np.zeros(local.shape[0], dtype=bool)
    selU[U] = True
    selF = np.zeros(local.shape[0], dtype=bool)
    selF[full] = True
    for l in range(spec.n_layers):
        if l == r0:
            Xf = round_store(np.asarray(boundary, dtype=np.float64)[full], spec.dtype)
            Xf[U - suffix_start] = X
            X = Xf
        if r0 <= l < r1:
            X = layer_rows(spec, weights[l], X, K[l], V[l], full,
                           _bias(local, sink, selF, alpha, beta, False))
        else:
            X = layer_rows(spec, weights[l], X, K[l], V[l], U,
                           _bias(local, sink, selU, alpha, beta, False))
        if l == r1 - 1:
            X = X[U - suffix_start]
    _commit(local, sink, U, False)
    return X, K, V, local, sink


# ----------------------------------------------------------------------------
# dense references used to build caches and to pin the recurrence
# ----------------------------------------------------------------------------

def prefill(spec: Spec, weights, X_in, block_bounds=None, return_boundary_at=None):
    """Ordinary causal prefill of a whole sequence X_in [N, d] at positions
    0..N-1.  block_bounds (half-open spans) restricts attention to the query's
    own block: independently prefilled blocks at their global positions
    ([KVX] Sec. 6.1-6.2).  Written as whole-sequence matrix algebra, separate
    from the packed-row code above.  Returns (X_out [N, d], K, V
    [L, H_kv, N, d_h]) and optionally the hidden state entering layer
    `return_boundary_at`."""
    rnd = lambda a: round_store(a, spec.dtype)
    Hq, Hkv, dh, F = spec.n_q_heads, spec.n_kv_heads, spec.head_dim, spec.ffn_dim
    G = Hq // Hkv
    X = rnd(np.asarray(X_in, dtype=np.float64))
    N = X.shape[0]
    allowed = np.tril(np.ones((N, N), dtype=bool))
    if block_bounds is not None:
        bid = np.full(N, -1)
        for i, (s, e) in enumerate(block_bounds):
            bid[s:e] = i
        allowed &= bid[:, None] == bid[None, :]
    pos = np.arange(N)
    Ks = np.zeros((spec.n_layers, Hkv, N, dh))
    Vs = np.zeros((spec.n_layers, Hkv, N, dh))
    boundary = None
    for l in range(spec.n_layers):
        if return_boundary_at == l:
            boundary = X.copy()
        W = weights[l]
        xn = rnd(rms_norm(X, W["norm1"], spec.rms_eps))
        qkv = xn @ W["w_qkv"].T
        if W.get("b_qkv") is not None:
            qkv = qkv + W["b_qkv"]
        q, k, v = qkv[:, :Hq * dh], qkv[:, Hq * dh:(Hq + Hkv) * dh], qkv[:, (Hq + Hkv) * dh:]
        if W.get("a_q") is not None:
            q = q + lora_delta(xn, W["a_q"], W["b_q"])
            v = v + lora_delta(xn, W["a_v"], W["b_v"])
        q, k = qk_norm(W, q.reshape(N, Hq, dh), k.reshape(N, Hkv, dh), spec.rms_eps)
        q = rnd(rope(q.transpose(1, 0, 2), pos, spec.rope_theta))
        k = rnd(rope(k.transpose(1, 0, 2), pos, spec.rope_theta))
        v = rnd(v.reshape(N, Hkv, dh).transpose(1, 0, 2))
        Ks[l], Vs[l] = k, v
        o = np.zeros((N, Hq, dh))
        for h in range(Hq):
            s = q[h] @ k[h // G].T / np.sqrt(dh)
            s[~allowed] = -np.inf
            p = np.exp(s - s.max(axis=1, keepdims=True))
            o[:, h, :] = (p / p.sum(axis=1, keepdims=True)) @ v[h // G]
        o = rnd(o).reshape(N, Hq * dh)
        hmid = X + o @ W["w_o"].T
        hn = rnd(rms_norm(hmid, W["norm2"], spec.rms_eps))
        gu = hn @ W["w_gate_up"].T
        act = rnd(silu(gu[:, :F]) * gu[:, F:])
        X = rnd(hmid + act @ W["w_down"].T)
    if return_boundary_at is not None:
        return X, Ks, Vs, boundary
    return X, Ks, Vs


def shift(K, V, start, d, theta):
    """Shift ([BKR] Sec. 7.1, Eq. 2): delete cache rows [start, start+d) and
    move the suffix down by d; keys are re-rotated by -d positions
    (R_{i-d} R_i^{-1} K_i), values move unchanged.  K, V [..., N, d_h]."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    N = K.shape[-2]
    n_move = N - start - d
    lead = K.shape[:-2]
    Kn = np.concatenate([K[..., :start, :], np.zeros(lead + (n_move, K.shape[-1]))], axis=-2)
    Vn = np.concatenate([V[..., :start, :], V[..., start + d:, :]], axis=-2)
    moved = K[..., start + d:, :].reshape(int(np.prod(lead)), n_move, K.shape[-1])
    rot = rope(moved, np.full(n_move, -d), theta)
    Kn[..., start:, :] = rot.reshape(lead + (n_move, K.shape[-1]))
    return Kn, Vn


def reposition(K, V, src_pos, dst_pos, theta):
    """Move a block computed on its own to new global positions ([NOTES]
    Sec. 5): keys stored after the rotary map at src_pos + i are re-rotated
    to dst_pos + i, i.e. rotated by dst_pos - src_pos; values carry no
    position and are returned as they are.  K, V [..., n, d_h]."""
    K = np.asarray(K, dtype=np.float64)
    n = K.shape[-2]
    flat = K.reshape(-1, n, K.shape[-1])
    Kn = rope(flat, np.full(n, float(dst_pos) - float(src_pos)), theta).reshape(K.shape)
    return Kn, np.asarray(V, dtype=np.float64).copy()


def attend(q, K_l, V_l, positions, local, sink, alpha, beta):
    """Inference mode of F ([KVX] Sec. 6.4): attention only, no write-back,
    with the stored correction masks.  q [B, Hq, d_h] for the sorted
    selected positions."""
    U = sorted_positions(positions)
    bias = alpha * np.asarray(local, dtype=np.float64) + beta * np.asarray(sink, dtype=np.float64)
    return attention(q, np.asarray(K_l, dtype=np.float64), np.asarray(V_l, dtype=np.float64), U, bias)
