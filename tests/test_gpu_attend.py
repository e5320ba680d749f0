"""GPU parity of the inference mode of operator F (kvr_attend: attention
only, stored correction masks, no write-back) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from selective_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup  # noqa: E402
from helpers import TOL, assert_close, f64, small_bf16  # noqa: E402


@pytest.mark.parametrize("dtype,alpha,beta", [("bf16", 0.0, 0.0), ("bf16", -2.0, -4.0), ("f32", -2.0, -4.0)])
def test_attend_matches_oracle(dtype, alpha, beta):
    if dtype == "bf16":
        w = small_bf16(n_layers=2, selection="isolated", n_select=200, alpha=alpha, beta=beta)
    else:
        base = wl.WORKLOADS["tiny"]
        import dataclasses
        w = dataclasses.replace(base, alpha=alpha, beta=beta, selection="isolated", n_select=300)
    rng = np.random.default_rng(3)
    local = rng.random((1, w.capacity)) < 0.5
    sink = rng.random((1, w.capacity)) < 0.2
    s = Setup(w, local=local, sink=sink)
    K_in = s.K.clone()
    s.select()
    R = s.n_rows
    m = w.model
    q = torch.randn(R, m.n_q_heads, m.head_dim, device="cuda").to(m.torch_dtype)
    out = torch.empty(R, m.n_q_heads * m.head_dim, device="cuda", dtype=m.torch_dtype)
    ws = torch.empty(kvr.kvr_workspace_bytes(s.handle, 0), dtype=torch.uint8, device="cuda")
    for layer in range(m.n_layers):
        want = oracle.attend(f64(q), f64(s.K[0, layer]), f64(s.V[0, layer]), s.positions[0],
                             local[0], sink[0], alpha, beta).reshape(R, -1)
        # without a workspace the kernel runs unsplit; with one it may split each
        # query tile's K/V range over several CTAs and merge their partials
        for workspace in (None, ws):
            out.zero_()
            kvr.kvr_attend(s.handle, layer, q, out, workspace, 0 if workspace is None else ws.numel())
            s.sync()
            assert_close(f64(out), want, TOL[dtype], f"attend layer {layer} workspace={workspace is not None}")
    assert torch.equal(s.K, K_in)
    s.close()
