"""kvr_refresh_layer_noalloc: the refresh layer for callers that cannot give
the library scratch memory (their device memory is owned by another
allocator, or they must not allocate after start-up).  It runs the same
kernels on the same plan as kvr_refresh_layer with a caller workspace, so its
results must be bit-identical to that entry point's, call after call, even
when the shared array still holds an earlier, larger call's data; and it must
reject a selection whose scratch exceeds its fixed 64 MiB array.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test."""
import dataclasses

import numpy as np
import pytest
import torch

from selective_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup  # noqa: E402
from helpers import small_bf16  # noqa: E402


def test_noalloc_matches_workspace_entry_point_two_calls():
    w = small_bf16(n_layers=2, selection="isolated", n_select=180, alpha=-2.0, beta=-4.0)
    rng = np.random.default_rng(21)
    local = rng.random((1, w.capacity)) < 0.5
    sink = rng.random((1, w.capacity)) < 0.2
    layers = wl.make_layer_weights(w, "cuda")
    # a larger selection on a third cache first: the shared array then holds
    # that call's data (its rows sit at other offsets) when the compared calls run
    big = dataclasses.replace(w, n_select=400)
    d = Setup(big, weights=layers, local=local, sink=sink)
    d.select()
    kvr.kvr_refresh_layer_noalloc(d.handle, 0, d.warr[0], d.hidden, 0)
    d.sync()
    d.close()
    a = Setup(w, weights=layers, local=local, sink=sink)   # caller workspace
    b = Setup(w, weights=layers, local=local, sink=sink)   # no-allocation variant
    assert torch.equal(a.K, b.K) and torch.equal(a.V, b.V)
    a.select()
    b.select()
    for layer in range(2):      # two calls in a row
        flags = kvr.KVR_COMMIT_META if layer == 1 else 0
        kvr.kvr_refresh_layer(a.handle, layer, a.warr[layer], a.hidden, a.ws, a.ws_bytes, flags)
        kvr.kvr_refresh_layer_noalloc(b.handle, layer, b.warr[layer], b.hidden, flags)
        a.sync()
        b.sync()
        assert torch.equal(b.hidden[:b.n_rows], a.hidden[:a.n_rows]), f"hidden after layer {layer}"
        assert torch.equal(b.K[0, layer], a.K[0, layer]), f"K layer {layer}"
        assert torch.equal(b.V[0, layer], a.V[0, layer]), f"V layer {layer}"
    la, sa = kvr.kvr_read_meta(a.handle, 1, a.words)
    lb, sb = kvr.kvr_read_meta(b.handle, 1, b.words)
    np.testing.assert_array_equal(la, lb)
    np.testing.assert_array_equal(sa, sb)
    a.close()
    b.close()


def test_noalloc_rejects_selection_beyond_its_scratch():
    base = wl.WORKLOADS["llama8b"]
    w = dataclasses.replace(base, model=dataclasses.replace(base.model, n_layers=1), n_select=1500,
                            selection="isolated")
    s = Setup(w)
    s.select()
    assert kvr.kvr_workspace_bytes(s.handle, 0) > (64 << 20)
    K_before = s.K.clone()
    with pytest.raises(kvr.KvrError) as e:
        kvr.kvr_refresh_layer_noalloc(s.handle, 0, s.warr[0], s.hidden, 0)
    assert e.value.status == kvr.KVR_EINVAL
    assert "64" in str(e.value) or "67108864" in str(e.value)
    s.sync()
    assert torch.equal(s.K, K_before)
    s.close()
