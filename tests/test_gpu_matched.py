"""The pages' matched-work geometry (Budgeted KV-Cache Repair for Evolving
Contexts, Sec. 13.3): a Qwen3-8B-shaped block (d 4096, 32/8 heads x 128, FFN
12288) cut to two layers so the oracle stays cheap, a prompt of 2056 tokens
that loses 8 at 64 (Shift), and 64 positions in R intervals with the M(U) the
pages state.  Layer 0's written K/V rows and the refreshed rows after layer
0 against the oracle (same Shift, same refresh), every other cache row
bit-identical to the shifted cache, the interval count and M(U) exact."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from selective_kv_cache_gb300 import workloads as wl

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup  # noqa: E402
from helpers import TOL, LazyWeights, assert_close, assert_close_rows, f64, oracle_spec  # noqa: E402


@pytest.mark.parametrize("R", [1, 16])
def test_matched_work_geometry_layer0(R):
    N, d_del, at = 2048, 8, 64
    base = wl.WORKLOADS["qwen3_matched"]
    m = dataclasses.replace(base.model, n_layers=2)
    w = dataclasses.replace(base, model=m, capacity=N + d_del, n_tokens=N + d_del, suffix_start=at)
    pos = wl.matched_positions(N, 64, R)
    assert int(np.sum(pos.astype(np.int64) + 1)) == 65568          # the pages' M(U) at 2K
    s = Setup(w, positions=[pos])
    K_in, V_in = s.K.clone(), s.V.clone()
    kvr.kvr_shift(s.handle, at, d_del)
    assert kvr.kvr_cache_info(s.handle) == (N, at)
    K_s, V_s = s.K.clone(), s.V.clone()
    rows, ivs = s.select()
    assert (rows, ivs) == (64, R)
    # layer 0 alone first (the refreshed rows X^1 depend on the inputs only);
    # the full run rewrites layer 0's selected rows before reading them
    s.refresh(0, 1, flags=0)
    s.sync()
    X1_gpu = f64(s.hidden[:64])
    s.select()
    s.refresh()
    s.sync()
    # oracle: the same Shift on the input cache, then layer 0 of the packed refresh
    spec = dataclasses.replace(oracle_spec(w), n_layers=1)
    K0, V0 = oracle.shift(f64(K_in[0, :1]), f64(V_in[0, :1]), at, d_del, m.rope_theta)
    U = oracle.sorted_positions(pos)
    ids = s.ids[0].cpu().numpy()
    X_src = np.zeros((N, m.d_model))
    X_src[U] = f64(s.embed[torch.from_numpy(ids[U].astype(np.int64)).cuda()])
    loc = oracle.shift_mask(s.local_mask[0], at, d_del)[:N]     # the bits moved with their tokens
    snk = oracle.shift_mask(s.sink_mask[0], at, d_del)[:N]
    X1, K, V, _, _ = oracle.refresh_packed(spec, LazyWeights(s.layers), K0, V0, loc, snk, U, X_src, 0.0, 0.0, False,
                                           n_layers=1)
    assert_close_rows(X1_gpu, X1, TOL["bf16"], "refreshed rows after layer 0")
    Ut = torch.from_numpy(U)
    assert_close(f64(s.K[0, 0][:, Ut]), K[0][:, U], TOL["bf16"], "K layer 0")
    assert_close(f64(s.V[0, 0][:, Ut]), V[0][:, U], TOL["bf16"], "V layer 0")
    keep = torch.ones(w.capacity, dtype=torch.bool, device="cuda")
    keep[Ut.cuda()] = False
    assert torch.equal(s.K[..., keep, :], K_s[..., keep, :])
    assert torch.equal(s.V[..., keep, :], V_s[..., keep, :])
    assert torch.isfinite(s.hidden[:64].float()).all()
    s.close()
