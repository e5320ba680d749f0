"""The two merges of a split attention -- by the last CTA of each query tile
inside the attention launch, or by a merge kernel after it -- write the same
output bits.  kvr_attend at the Llama-3-8B (units and isolated positions),
block-seam and matched-work shapes under KVR_ATTN_MERGE=cta and =kernel, the
kernel merge also against the oracle; and a two-layer Llama-3-8B refresh
under both, its hidden rows and cache bit for bit."""
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from selective_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup  # noqa: E402
from helpers import TOL, assert_close, assert_rel_heads, f64  # noqa: E402


# K/V tiles per CTA, pinned so that both merges see the same split: the
# longest query tile's range in 4 (Llama-3-8B: 60 tiles), 3 (seam: 128) or up
# to 16 (matched work: 64) chunks
CHUNK = {"llama8b": 16, "llama8b_frag": 16, "qwen7b_seam": 48, "qwen3_matched": 4}


def _with_merge(mode, chunk, fn):
    env = {"KVR_ATTN_MERGE": mode, "KVR_ATTN_CHUNK": str(chunk)}
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        return fn()
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


def _layers(name, n):
    base = wl.WORKLOADS[name]
    return dataclasses.replace(base, model=dataclasses.replace(base.model, n_layers=n))


@pytest.mark.parametrize("name", ["llama8b", "llama8b_frag", "qwen7b_seam", "qwen3_matched"])
def test_attend_merges_write_the_same_bits(name):
    w = _layers(name, 1)
    s = Setup(w)
    m = w.model
    g = torch.Generator(device="cuda").manual_seed(17)
    outs, launches = {}, {}
    for mode in ("cta", "kernel"):
        def run():
            s.select()
            R = s.n_rows
            q = torch.randn(R, m.n_q_heads, m.head_dim, device="cuda", generator=g.manual_seed(17)).to(m.torch_dtype)
            out = torch.full((R, m.n_q_heads * m.head_dim), float("nan"), device="cuda", dtype=m.torch_dtype)
            ws = torch.empty(kvr.kvr_workspace_bytes(s.handle, 0), dtype=torch.uint8, device="cuda")
            kvr.kvr_profile_enable(s.handle, True)
            kvr.kvr_attend(s.handle, 0, q, out, ws, ws.numel())
            s.sync()
            n = kvr.kvr_profile_read(s.handle)["attention"][0]
            kvr.kvr_profile_enable(s.handle, False)
            return q, out, n
        q, outs[mode], launches[mode] = _with_merge(mode, CHUNK[name], run)
    assert launches == {"cta": 1, "kernel": 2}, launches   # the kernel merge ran, so the range was split
    assert torch.isfinite(outs["kernel"].float()).all()
    assert torch.equal(outs["cta"], outs["kernel"])
    if name in ("llama8b", "qwen3_matched"):   # oracle rows: all of them at these row counts
        want = oracle.attend(f64(q), f64(s.K[0, 0]), f64(s.V[0, 0]), s.positions[0], s.local_mask[0],
                             s.sink_mask[0], w.alpha, w.beta).reshape(s.n_rows, -1)
        assert_close(f64(outs["kernel"]), want, TOL["bf16"], f"{name} merge kernel")
        assert_rel_heads(f64(outs["kernel"]), want, TOL["bf16"], m.head_dim, f"{name} merge kernel")
    s.close()


@pytest.mark.slow
def test_refresh_merges_write_the_same_bits():
    w = _layers("llama8b", 2)
    res = {}
    for mode in ("cta", "kernel"):
        def run():
            s = Setup(w)
            s.select()
            s.refresh()
            s.sync()
            r = (s.hidden[:s.n_rows].clone(), s.K.clone(), s.V.clone())
            s.close()
            return r
        res[mode] = _with_merge(mode, CHUNK["llama8b"], run)
    for a, b, what in zip(res["cta"], res["kernel"], ("hidden", "K", "V")):
        assert torch.equal(a, b), what
    assert np.isfinite(f64(res["kernel"][0])).all()
