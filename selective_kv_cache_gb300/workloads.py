"""Seeded synthetic inputs for selective KV-cache refresh.

This module only draws random numbers and lays them out.  It holds none of
the refresh arithmetic (no norm, projection, rotary map or attention): both
the CPU oracle and the CUDA path receive the tensors built here, and neither
computes anything here.

Workloads (all synthetic, random-init weights; the pages evaluate on trained
checkpoints and text datasets that are not available here):

  tiny      1 layer, d=256, 4x64 MHA, FFN 1024, fp32, N=1024, prefix 0..255
            valid, 4 units of 16 positions, alpha=beta=0.
  llama8b   Llama-3-8B shape (32 L, 4096, 32/8 x 128, FFN 14336,
            theta 5e5), bf16; 8192 tokens, 512 deleted at 2048 -> N=7680,
            P=2048, S=5632; 5 % budget = 282 positions in units of 32-64.
  llama8b_frag  same model and edit; 282 isolated positions (fragmented).
  qwen7b_seam   Qwen2.5-7B shape (28 L, 3584, 28/4 x 128, FFN 18944), bf16;
            N=16384 as 8 blocks of 2048; seam windows tau=64 with the
            asymmetric first-seam rule; alpha=-2, beta=-4; sinks 0..3.
  qwen1p5b_drift Qwen2.5-1.5B shape (28 L, 1536, 12/2 x 128, FFN 8960), bf16,
            batch 4 x 32768; layers 10..14 over the whole suffix
            [8192, 32768), 492 isolated positions elsewhere; rank-16 LoRA
            on Q and V.

Seeds: base 20261202 + 100*k for workload k, sub-streams +0 weights,
+1 tokens/hidden, +2 dirty perturbation, +3 selection, +4/+5 adapters,
+6 cache contents.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    rope_theta: float
    rms_eps: float
    dtype: str          # "f32" or "bf16"
    qkv_bias: bool
    vocab: int = 32000
    qk_norm: bool = False   # Qwen3: RMSNorm of every Q and K head before RoPE

    @property
    def qkv_out(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    model: ModelShape
    batch: int
    capacity: int        # cache rows per sequence
    n_tokens: int        # valid cache length after the edit
    suffix_start: int    # retained prefix [0, suffix_start) is valid
    n_select: int        # positions refreshed per sequence
    alpha: float = 0.0
    beta: float = 0.0
    selection: str = "units"   # units | isolated | seams | range
    range_layers: tuple = ()   # (r0, r1): layers recomputed over the whole suffix
    lora_rank: int = 0
    uses_embeddings: bool = True
    n_intervals: int = 0       # "matched" selection: the interval count R

    def seed(self, stream: int) -> int:
        return BASE_SEED + 100 * self.index + stream


TINY = ModelShape(1, 256, 4, 4, 64, 1024, 10000.0, 1e-5, "f32", False)
LLAMA8B = ModelShape(32, 4096, 32, 8, 128, 14336, 500000.0, 1e-5, "bf16", False)
QWEN7B = ModelShape(28, 3584, 28, 4, 128, 18944, 1000000.0, 1e-6, "bf16", True)
# Qwen3-8B geometry (36 layers, hidden 4096, 32 query / 8 K/V heads x 128, FFN
# 12288, vocabulary 151936): the model of the pages' matched-work benchmark
# ("Budgeted KV-Cache Repair for Evolving Contexts", Sec. 13.3).
QWEN3_8B = ModelShape(36, 4096, 32, 8, 128, 12288, 1000000.0, 1e-6, "bf16", False, vocab=151936, qk_norm=True)
QWEN1P5B = ModelShape(28, 1536, 12, 2, 128, 8960, 1000000.0, 1e-6, "bf16", True)

WORKLOADS = {
    "tiny": Workload("tiny", 0, TINY, 1, 1024, 1024, 256, 64,
                     selection="units", uses_embeddings=False),
    # Budget B(S, b) = min(S, ceil(S*b/100)) with S = 5632, b = 5 gives 282
    # ("Budgeted KV-Cache Repair for Evolving Contexts", Sec. 7.1, Eq. 3).
    "llama8b": Workload("llama8b", 1, LLAMA8B, 1, 8192, 7680, 2048, 282,
                        selection="units"),
    "llama8b_frag": Workload("llama8b_frag", 2, LLAMA8B, 1, 8192, 7680, 2048, 282,
                             selection="isolated"),
    "qwen7b_seam": Workload("qwen7b_seam", 3, QWEN7B, 1, 16384, 16384, 0, 896,
                            alpha=-2.0, beta=-4.0, selection="seams"),
    "qwen1p5b_drift": Workload("qwen1p5b_drift", 4, QWEN1P5B, 4, 32768, 32768, 8192, 492,
                               selection="isolated", range_layers=(10, 15), lora_rank=16),
    # the pages' matched-work benchmark: 8200-token prompt, 8 tokens deleted at
    # 64 (Shift), 64 positions in 16 intervals about the centre of the 8192
    # remaining (the bench runs N in {2048, 8192} and R in {1, 4, 16})
    "qwen3_matched": Workload("qwen3_matched", 9, QWEN3_8B, 1, 8200, 8192, 64, 64, selection="matched",
                              n_intervals=16),
    # the Llama-3-8B-shaped refresh cut to 2 layers: a small case (about 1.2 GB
    # on the device) for kernel profiles of the same launch configuration
    "llama8b_2l": Workload("llama8b_2l", 1, dataclasses.replace(LLAMA8B, n_layers=2), 1, 8192, 7680, 2048, 282,
                           selection="units"),
}


def shrink(w: Workload, *, n_layers=None, d_model=None, n_q_heads=None, n_kv_heads=None,
           ffn_dim=None, capacity=None, n_tokens=None, suffix_start=None, n_select=None,
           batch=None, name=None) -> Workload:
    """A smaller copy of a workload (same structure) for fast parity tests."""
    m = w.model
    m2 = dataclasses.replace(
        m,
        n_layers=n_layers or m.n_layers, d_model=d_model or m.d_model,
        n_q_heads=n_q_heads or m.n_q_heads, n_kv_heads=n_kv_heads or m.n_kv_heads,
        ffn_dim=ffn_dim or m.ffn_dim)
    return dataclasses.replace(
        w, name=name or (w.name + "_small"), model=m2,
        capacity=capacity or w.capacity, n_tokens=n_tokens or w.n_tokens,
        suffix_start=w.suffix_start if suffix_start is None else suffix_start,
        n_select=n_select or w.n_select, batch=batch or w.batch)


# ----------------------------------------------------------------------------
# random tensors
# ----------------------------------------------------------------------------

def _normal(shape, std, seed, device, out_dtype, rng_state=None):
    """N(0, std^2) in fp32, cast to out_dtype (round-to-nearest-even)."""
    if device == "cpu":
        rng = rng_state if rng_state is not None else np.random.Generator(np.random.PCG64(seed))
        a = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)
        return torch.from_numpy(a).to(out_dtype)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t.to(out_dtype)


def make_layer_weights(w: Workload, device="cpu", lora: Optional[str] = None):
    """Per-layer weights in nn.Linear layout ([out_features, in_features]).

    w_qkv     [(Hq + 2 Hkv) dh, d]  rows: Q heads, then K heads, then V heads
    b_qkv     [(Hq + 2 Hkv) dh] or None
    w_o       [d, Hq dh]
    w_gate_up [2F, d]               rows 0..F-1 gate, F..2F-1 up
    w_down    [d, F]
    norm1/2   [d]                    ones
    q_norm/k_norm [dh]               1 + 0.1 N(0, 1), only for shapes with qk_norm
    LoRA (lora='old'|'new'): a_q [r, d], b_q [Hq dh, r], a_v [r, d], b_v [Hkv dh, r]
    """
    m = w.model
    dt = m.torch_dtype
    base = w.seed(0)
    layers = []
    for l in range(m.n_layers):
        s = base * 1000 + 17 * l
        rng = np.random.Generator(np.random.PCG64(s)) if device == "cpu" else None
        L = {
            "w_qkv": _normal((m.qkv_out, m.d_model), 0.02, s + 1, device, dt, rng),
            "b_qkv": _normal((m.qkv_out,), 0.02, s + 2, device, dt, rng) if m.qkv_bias else None,
            "w_o": _normal((m.d_model, m.n_q_heads * m.head_dim), 0.02, s + 3, device, dt, rng),
            "w_gate_up": _normal((2 * m.ffn_dim, m.d_model), 0.02, s + 4, device, dt, rng),
            "w_down": _normal((m.d_model, m.ffn_dim), 0.02, s + 5, device, dt, rng),
            "norm1": torch.ones(m.d_model, dtype=dt, device=device),
            "norm2": torch.ones(m.d_model, dtype=dt, device=device),
        }
        if m.qk_norm:
            L["q_norm"] = (1.0 + _normal((m.head_dim,), 0.1, s + 6, device, torch.float32, rng)).to(dt)
            L["k_norm"] = (1.0 + _normal((m.head_dim,), 0.1, s + 7, device, torch.float32, rng)).to(dt)
        if lora is not None and w.lora_rank > 0:
            ls = w.seed(4 if lora == "old" else 5) * 1000 + 17 * l
            lrng = np.random.Generator(np.random.PCG64(ls)) if device == "cpu" else None
            r = w.lora_rank
            L["a_q"] = _normal((r, m.d_model), 0.01, ls + 1, device, dt, lrng)
            L["b_q"] = _normal((m.n_q_heads * m.head_dim, r), 0.01, ls + 2, device, dt, lrng)
            L["a_v"] = _normal((r, m.d_model), 0.01, ls + 3, device, dt, lrng)
            L["b_v"] = _normal((m.n_kv_heads * m.head_dim, r), 0.01, ls + 4, device, dt, lrng)
        layers.append(L)
    return layers


def make_embeddings(w: Workload, device="cpu"):
    """Embedding table [vocab, d] ~ N(0, 1) in model dtype."""
    m = w.model
    return _normal((m.vocab, m.d_model), 1.0, w.seed(1) * 1000 + 1, device, m.torch_dtype)


def make_token_ids(w: Workload, device="cpu"):
    """Token ids [batch, capacity] uniform over [0, vocab) (int32)."""
    rng = np.random.Generator(np.random.PCG64(w.seed(1)))
    ids = rng.integers(0, w.model.vocab, size=(w.batch, w.capacity), dtype=np.int64)
    return torch.from_numpy(ids.astype(np.int32)).to(device)


def make_hidden_inputs(w: Workload, device="cpu", dirty=False):
    """Per-position hidden inputs [batch, capacity, d] ~ N(0, 1) (tiny workload).

    dirty=True adds 0.5 * N(0, 1) on the retained suffix: the stale context the
    cache was built from before the edit."""
    m = w.model
    rng = np.random.Generator(np.random.PCG64(w.seed(1)))
    h = rng.standard_normal(size=(w.batch, w.capacity, m.d_model), dtype=np.float32)
    if dirty:
        rng2 = np.random.Generator(np.random.PCG64(w.seed(2)))
        p = rng2.standard_normal(size=h.shape, dtype=np.float32)
        h[:, w.suffix_start:, :] += np.float32(0.5) * p[:, w.suffix_start:, :]
    return torch.from_numpy(h).to(m.torch_dtype).to(device)


def make_random_cache(w: Workload, device="cpu", std=1.0):
    """Stale K/V ~ N(0, std^2) in model dtype, layout [batch, L, Hkv, capacity, dh]."""
    m = w.model
    shape = (w.batch, m.n_layers, m.n_kv_heads, w.capacity, m.head_dim)
    k = _normal(shape, std, w.seed(6) * 1000 + 1, device, m.torch_dtype)
    v = _normal(shape, std, w.seed(6) * 1000 + 2, device, m.torch_dtype)
    return k, v


# ----------------------------------------------------------------------------
# selections and metadata
# ----------------------------------------------------------------------------

def _units(rng, lo, hi, count, len_lo, len_hi):
    """Non-overlapping contiguous units in [lo, hi) until `count` positions are
    taken; the last unit keeps only its first positions (units may touch)."""
    taken = np.zeros(hi, dtype=bool)
    out = []
    remaining = count
    tries = 0
    while remaining > 0:
        tries += 1
        if tries > 100000:
            raise RuntimeError("unit placement failed")
        ln = int(rng.integers(len_lo, len_hi + 1))
        st = int(rng.integers(lo, hi - ln + 1))
        if taken[st:st + ln].any():
            continue
        take = min(ln, remaining)
        taken[st:st + ln] = True
        out.extend(range(st, st + take))
        remaining -= take
    return out


def make_positions(w: Workload):
    """Selected positions per sequence, in the order the generator draws them
    (NOT sorted: sorting is the selection step's job).  Returns a list of
    int32 arrays, one per sequence."""
    rng = np.random.Generator(np.random.PCG64(w.seed(3)))
    lo, hi = w.suffix_start, w.n_tokens
    seqs = []
    for _ in range(w.batch):
        if w.selection == "units":
            if w.model.dtype == "f32":     # tiny: 4 units of 16
                pos = _units(rng, lo, hi, w.n_select, 16, 16)
            else:                          # units of 32..64 tokens
                pos = _units(rng, lo, hi, w.n_select, 32, 64)
        elif w.selection == "isolated":
            pos = (rng.choice(hi - lo, size=w.n_select, replace=False) + lo).tolist()
        elif w.selection == "seams":
            pos = seam_positions(w)
        elif w.selection == "matched":
            pos = matched_positions(w.n_tokens, w.n_select, w.n_intervals).tolist()
        elif w.selection == "all":
            pos = list(range(lo, hi))
        else:
            raise ValueError(w.selection)
        pos = np.array(pos, dtype=np.int32)
        rng.shuffle(pos)
        seqs.append(pos)
    return seqs


def make_unit_bounds(S: int, seed: int, lo: int = 8, hi: int = 128):
    """A synthetic partition of an S-token suffix into semantic units of lo..hi
    tokens (text segmentation stands outside the method's hot path): int32
    offsets 0 = b_0 < ... < b_n = S.  The last unit takes the remainder and
    may be shorter than lo."""
    rng = np.random.Generator(np.random.PCG64(seed))
    b = [0]
    while b[-1] < S:
        b.append(min(S, b[-1] + int(rng.integers(lo, hi + 1))))
    return np.array(b, dtype=np.int32)


def make_query_ids(vocab: int, Q: int, seed: int, suffix_ids=None, overlap: int = 4):
    """Q query token ids, uniform over the vocabulary; `overlap` of them are
    copied from the suffix so that the identical-token bonus occurs."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.integers(0, vocab, size=Q).astype(np.int32)
    if suffix_ids is not None and overlap > 0:
        sid = np.asarray(suffix_ids)
        q[:overlap] = sid[rng.integers(0, sid.size, size=overlap)]
    return q


def matched_positions(N: int, B: int, R: int, spacing: int = 64):
    """The matched-work geometry of the pages' execution benchmark ("Budgeted
    KV-Cache Repair for Evolving Contexts", Sec. 13.3, Table 18): B positions
    as R intervals of B/R tokens placed symmetrically about the centre
    (N - 1)/2, so M(U) = sum(u + 1) = B (N + 1) / 2 is the same for every R
    (65,568 at N = 2048 and 262,176 at N = 8192 with B = 64, the values the
    pages state).  Interval k spans [a_k, a_k + B/R) with mean
    (N - 1)/2 + (k - (R - 1)/2) * spacing; an even spacing keeps every a_k
    an integer."""
    L = B // R
    assert L * R == B and spacing >= L and spacing % 2 == 0
    c = (N - 1) / 2.0
    starts = [c - (L - 1) / 2.0 + (k - (R - 1) / 2.0) * spacing for k in range(R)]
    assert all(float(x).is_integer() for x in starts)
    pos = np.concatenate([np.arange(int(a), int(a) + L) for a in starts])
    assert pos.min() >= 0 and pos.max() < N
    return pos.astype(np.int32)


def block_bounds(w: Workload, n_blocks=8):
    """Half-open block spans [s_i, e_i) of an equal-block layout."""
    size = w.n_tokens // n_blocks
    return [(i * size, (i + 1) * size) for i in range(n_blocks)]


def seam_positions(w: Workload, tau=64, n_blocks=8):
    """Seam windows at every block boundary; at the first seam the window
    covers only the head of block 2, and the unused tau goes to the tail of
    the last block (the asymmetric rule)."""
    b = block_bounds(w, n_blocks)
    pos = set()
    for i in range(len(b) - 1):
        (s0, e0), (s1, e1) = b[i], b[i + 1]
        if i > 0:
            pos.update(range(max(s0, e0 - tau), e0))
        pos.update(range(s1, min(e1, s1 + tau)))
    s_last, e_last = b[-1]
    pos.update(range(max(s_last, e_last - tau), e_last))
    return sorted(pos)


def make_metadata(w: Workload):
    """(local, sink) boolean arrays [batch, capacity].

    Retained-prefix positions are global; stale positions are local.  For the
    block-seam workload, block 1 is global and blocks 2..m are local, and the
    first 4 positions of blocks 2..m are the spurious sinks S' (the true sinks
    0..3 at sequence start are never penalised)."""
    local = np.zeros((w.batch, w.capacity), dtype=bool)
    sink = np.zeros((w.batch, w.capacity), dtype=bool)
    if w.selection == "seams":
        b = block_bounds(w)
        local[:, b[1][0]:w.n_tokens] = True
        for (s, e) in b[1:]:
            sink[:, s:s + 4] = True
    else:
        local[:, w.suffix_start:w.n_tokens] = True
    return local, sink


def pack_bits(mask: np.ndarray) -> np.ndarray:
    """Bool [..., n] -> uint32 words [..., ceil(n/32)], bit b of word w is
    element 32*w + b."""
    n = mask.shape[-1]
    nw = (n + 31) // 32
    pad = np.zeros(mask.shape[:-1] + (nw * 32,), dtype=np.uint64)
    pad[..., :n] = mask
    pad = pad.reshape(mask.shape[:-1] + (nw, 32))
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (pad * weights).sum(axis=-1).astype(np.uint32)
