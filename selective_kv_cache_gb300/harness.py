"""Device-side set-up of a refresh workload: allocates the weights, cache,
metadata and row sources with torch, binds them to a libkvr cache handle and
drives the C entry points.  Shared by the GPU tests and bench.py; it holds
none of the method's arithmetic (that runs in libkvr's kernels)."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import kvr
from . import workloads as wl


def merge_lora(layers, shape, stream=None):
    """Fold each layer's LoRA (a_q/b_q on the Q rows, a_v/b_v on the V rows of
    w_qkv) into a new w_qkv with kvr_lora_merge; returns new layer dicts."""
    out = []
    dt = kvr.KVR_BF16 if shape.dtype == "bf16" else kvr.KVR_F32
    hq, hkv, dh, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.d_model
    for L in layers:
        M = dict(L)
        if L.get("a_q") is not None:
            wq = torch.empty_like(L["w_qkv"])
            r = L["a_q"].shape[0]
            kvr.kvr_lora_merge(L["w_qkv"], wq, shape.qkv_out, d, 0, hq * dh, L["a_q"], L["b_q"], r, 1.0, dt, stream)
            kvr.kvr_lora_merge(wq, wq, shape.qkv_out, d, (hq + hkv) * dh, hkv * dh, L["a_v"], L["b_v"], r, 1.0, dt,
                               stream)
            M["w_qkv"] = wq
        out.append(M)
    return out


def pack_adapter(layers):
    """The adapter as one flat parameter vector theta: every layer's a_q, b_q,
    a_v, b_v flattened and concatenated in layer order (the layout the
    layer-range policy takes)."""
    parts = []
    for L in layers:
        for k in ("a_q", "b_q", "a_v", "b_v"):
            if L.get(k) is not None:
                parts.append(L[k].reshape(-1))
    return torch.cat(parts)


def shard_sequences(batch: int, world: int, rank: int):
    """Sequences [lo, hi) of a batch that rank `rank` of `world` owns: the
    sequences are independent problems (own cache, own selection), so they
    split into contiguous, near-equal shards with no exchange between ranks;
    the first batch % world ranks take one more."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    base, extra = divmod(batch, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


class Setup:
    """One workload bound to a libkvr cache on the current CUDA device.

    cache: "random" (seeded N(0, 1) K/V) or a (K, V) pair of device tensors in
    the [batch, L, H_kv, capacity, d_h] layout.  positions: override of the
    selection (list of int arrays, one per sequence)."""

    def __init__(self, w: wl.Workload, cache="random", positions=None, weights=None, flags=0,
                 local=None, sink=None, device="cuda", embed=None, seqs=None):
        # seqs = (lo, hi): bind only sequences [lo, hi) of the workload's batch
        # (a rank's shard); their inputs are the full batch's, sliced
        full = w
        lo, hi = (0, w.batch) if seqs is None else seqs
        if seqs is not None:
            w = dataclasses.replace(w, batch=hi - lo)
        self.seqs = (lo, hi)
        self.w = w
        self.shape = w.model
        self.device = device
        self.layers = weights if weights is not None else wl.make_layer_weights(w, device)
        self.warr = kvr.layer_weights_array(self.layers)
        if isinstance(cache, str):
            K, V = wl.make_random_cache(full, device)
            self.K, self.V = (K, V) if seqs is None else (K[lo:hi].clone(), V[lo:hi].clone())
            del K, V
        else:
            self.K, self.V = cache
        lm, sm = wl.make_metadata(full)
        lm, sm = lm[lo:hi], sm[lo:hi]
        if local is not None:
            lm = local
        if sink is not None:
            sm = sink
        self.local_mask, self.sink_mask = lm, sm
        self.flags = flags
        self.handle = kvr.kvr_create_cache(
            kvr.model_desc(self.shape), w.batch, w.capacity, self.K, self.V, w.n_tokens, w.suffix_start,
            np.ascontiguousarray(wl.pack_bits(lm)), np.ascontiguousarray(wl.pack_bits(sm)),
            w.alpha, w.beta, flags)
        self.words = (w.capacity + 31) // 32
        if w.uses_embeddings:
            self.embed = embed if embed is not None else wl.make_embeddings(w, device)
            self.ids = wl.make_token_ids(full, device)[lo:hi].contiguous()
            self.hidden_src = None
        else:
            self.embed = self.ids = None
            self.hidden_src = wl.make_hidden_inputs(full, device)[lo:hi].contiguous()
        self.positions = positions if positions is not None else wl.make_positions(full)[lo:hi]
        self.pos_host = np.ascontiguousarray(np.concatenate(self.positions).astype(np.int32))
        self.counts = np.array([len(p) for p in self.positions], np.int32)
        self.n_rows = int(self.counts.sum())
        self.hidden = torch.empty((max(self.n_rows, 1), self.shape.d_model), dtype=self.shape.torch_dtype,
                                  device=device)
        self.ws_bytes = 0
        self.ws = None

    def select(self, budget_percent=-1, stream=None):
        n = int(np.asarray(self.counts).sum())
        if n > self.hidden.shape[0]:
            self.hidden = torch.empty((n, self.shape.d_model), dtype=self.shape.torch_dtype, device=self.device)
        self.n_rows = n
        rows, ivs = kvr.kvr_select(
            self.handle, self.pos_host, self.counts, budget_percent,
            token_ids=self.ids, embed_table=self.embed, vocab=self.shape.vocab if self.embed is not None else 0,
            hidden_src=self.hidden_src, hidden_out=self.hidden, stream=stream)
        need = kvr.kvr_workspace_bytes(self.handle, 0)
        if self.ws is None or need > self.ws_bytes:
            self.ws_bytes = max(need, 256)
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        return rows, ivs

    def refresh(self, layer_begin=0, layer_end=None, flags=kvr.KVR_COMMIT_META, stream=None):
        L = self.shape.n_layers if layer_end is None else layer_end
        kvr.kvr_refresh(self.handle, self.warr, layer_begin, L, self.hidden, self.ws, self.ws_bytes, flags,
                        stream=stream)

    def refresh_interval_wise(self, layer_begin=0, layer_end=None, flags=kvr.KVR_COMMIT_META, stream=None):
        """The interval-major comparator over the same selection: returns the
        number of intervals.  Rows land in self.hidden in sorted order."""
        L = self.shape.n_layers if layer_end is None else layer_end
        longest = 1
        for pos in self.positions:
            u = np.sort(pos)
            run = 1
            for k in range(1, len(u)):
                run = run + 1 if u[k] == u[k - 1] + 1 else 1
                longest = max(longest, run)
        n = int(np.asarray(self.counts).sum())
        if n > self.hidden.shape[0]:
            self.hidden = torch.empty((n, self.shape.d_model), dtype=self.shape.torch_dtype, device=self.device)
        need = kvr.kvr_workspace_bytes(self.handle, max(longest, 1))
        if self.ws is None or need > self.ws_bytes:
            self.ws_bytes = need
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        return kvr.kvr_refresh_interval_wise(
            self.handle, self.pos_host, self.counts, -1, token_ids=self.ids, embed_table=self.embed,
            vocab=self.shape.vocab if self.embed is not None else 0, hidden_src=self.hidden_src,
            weights_array=self.warr, layer_begin=layer_begin, layer_end=L, hidden_out=self.hidden,
            workspace=self.ws, ws_bytes=self.ws_bytes, flags=flags, stream=stream)

    def refresh_range(self, boundary, r0, r1, stream=None):
        """Adapter-drift recovery through kvr_refresh_range: the selected rows
        through layers [0, r0), the whole affected suffix through [r0, r1)
        (rows not selected enter from `boundary` [batch, capacity, d], the
        stored hidden states at layer r0), then the selected rows again through
        [r1, L) and the commit."""
        w = self.w
        n_full = w.batch * (w.n_tokens - w.suffix_start)
        if getattr(self, "hidden_full", None) is None or self.hidden_full.shape[0] < n_full:
            self.hidden_full = torch.empty((n_full, self.shape.d_model), dtype=self.shape.torch_dtype,
                                           device=self.device)
        n = int(np.asarray(self.counts).sum())
        if n > self.hidden.shape[0]:
            self.hidden = torch.empty((n, self.shape.d_model), dtype=self.shape.torch_dtype, device=self.device)
        self.n_rows = n
        need = kvr.kvr_workspace_bytes(self.handle, n_full)
        if self.ws is None or need > self.ws_bytes:
            self.ws_bytes = need
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        kvr.kvr_refresh_range(self.handle, self.warr, r0, r1, self.pos_host, self.counts, token_ids=self.ids,
                              embed_table=self.embed, vocab=self.shape.vocab if self.embed is not None else 0,
                              hidden_src=self.hidden_src, boundary=boundary, hidden_sel=self.hidden,
                              hidden_full=self.hidden_full, workspace=self.ws, ws_bytes=self.ws_bytes,
                              flags=kvr.KVR_COMMIT_META, stream=stream)

    def sync(self, stream=None):
        kvr.kvr_sync_status(self.handle, stream)

    def close(self):
        if self.handle:
            kvr.kvr_destroy_cache(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
