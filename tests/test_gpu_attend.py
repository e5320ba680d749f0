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
from helpers import TOL, assert_close, assert_rel_heads, f64, small_bf16  # noqa: E402


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
            assert_rel_heads(f64(out), want, TOL[dtype], m.head_dim, f"attend layer {layer}")
    assert torch.equal(s.K, K_in)
    s.close()


@pytest.mark.slow
def test_attend_block_seam_full_shape():
    """kvr_attend at the block-seam workload's full attention shape: N = 16384
    in 8 blocks, the 896 seam rows, 28 query / 4 K/V heads x 128 (7 query
    heads per K/V head), alpha = -2, beta = -4 with the stored masks (blocks
    2..8 local, their first 4 positions the sinks S'), against the oracle on
    every row and head, without a workspace (each CTA walks a query tile's
    whole K/V range) and with one (split ranges merged afterwards)."""
    import dataclasses
    base = wl.WORKLOADS["qwen7b_seam"]
    w = dataclasses.replace(base, model=dataclasses.replace(base.model, n_layers=1))
    s = Setup(w)
    rows, ivs = s.select()
    assert (rows, ivs) == (896, 8)
    m = w.model
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn(rows, m.n_q_heads, m.head_dim, device="cuda", generator=g).to(m.torch_dtype)
    out = torch.empty(rows, m.n_q_heads * m.head_dim, device="cuda", dtype=m.torch_dtype)
    ws = torch.empty(kvr.kvr_workspace_bytes(s.handle, 0), dtype=torch.uint8, device="cuda")
    want = oracle.attend(f64(q), f64(s.K[0, 0]), f64(s.V[0, 0]), s.positions[0], s.local_mask[0], s.sink_mask[0],
                         w.alpha, w.beta).reshape(rows, -1)
    for workspace in (None, ws):
        out.zero_()
        kvr.kvr_attend(s.handle, 0, q, out, workspace, 0 if workspace is None else ws.numel())
        s.sync()
        assert_close(f64(out), want, TOL["bf16"], f"attend, workspace={workspace is not None}")
        assert_rel_heads(f64(out), want, TOL["bf16"], m.head_dim, f"attend, workspace={workspace is not None}")
    s.close()


def _tile_jumps(q, K, U, bias, G, keys_per_tile=128):
    """Per query row and head: the largest rise of the base-2 running maximum
    of the biased logits from one 128-key tile to the next (the walk a CTA
    makes over a query tile's K/V range from tile 0)."""
    R, Hq, dh = q.shape
    jumps = np.zeros((R, Hq))
    for r in range(R):
        n = int(U[r]) + 1
        for h in range(Hq):
            s = (K[h // G, :n] @ q[r, h]) / np.sqrt(dh) + bias[:n]
            x = s * np.log2(np.e)
            run = -np.inf
            for t0 in range(0, n, keys_per_tile):
                mt = x[t0:t0 + keys_per_tile].max()
                if t0 > 0:
                    jumps[r, h] = max(jumps[r, h], mt - run)
                run = max(run, mt)
    return jumps


@pytest.mark.parametrize("kind", ["late_local_bias", "aligned_key"])
def test_attend_peaked_softmax_rescales_output(kind):
    """A peaked softmax whose running maximum rises by more than 2^8 (base 2)
    after the first K/V tile, which makes the kernel rescale its output
    accumulator in tensor memory.  late_local_bias: alpha = +16 on local keys
    that exist only from position 400 on, and beta = +8 on sinks from 1000 on
    (two rises for the later rows); aligned_key: every query is 1.5 x the key
    three positions before its own, so its last tile holds one dominant key.
    Checked against the oracle without and with a workspace (split K/V
    ranges, whose chunks start their own running maxima)."""
    if kind == "late_local_bias":
        w = small_bf16(n_layers=1, selection="isolated", n_select=200, alpha=16.0, beta=8.0)
    else:
        w = small_bf16(n_layers=1, selection="isolated", n_select=200)
    local = np.zeros((1, w.capacity), bool)
    sink = np.zeros((1, w.capacity), bool)
    if kind == "late_local_bias":
        local[0, 400:w.n_tokens] = True
        sink[0, 1000:w.n_tokens:7] = True
    s = Setup(w, local=local, sink=sink)
    s.select()
    R = s.n_rows
    m = w.model
    G = m.n_q_heads // m.n_kv_heads
    U = np.sort(s.positions[0]).astype(np.int64)
    if kind == "late_local_bias":
        g = torch.Generator(device="cuda").manual_seed(9)
        q = torch.randn(R, m.n_q_heads, m.head_dim, device="cuda", generator=g).to(m.torch_dtype)
    else:
        kv = torch.arange(m.n_q_heads, device="cuda") // G
        src = torch.from_numpy(U - 3).cuda()
        q = (1.5 * s.K[0, 0][kv[None, :], src[:, None]].float()).to(m.torch_dtype)   # [R, Hq, dh]
    bias = w.alpha * local[0] + w.beta * sink[0]
    Kf, Vf = f64(s.K[0, 0]), f64(s.V[0, 0])
    jumps = _tile_jumps(f64(q), Kf, U, bias, G)
    assert (jumps > 8.0).mean() > 0.5, "the case must raise the running maximum by more than 2^8 after a tile"
    want = oracle.attend(f64(q), Kf, Vf, s.positions[0], local[0], sink[0], w.alpha, w.beta).reshape(R, -1)
    out = torch.empty(R, m.n_q_heads * m.head_dim, device="cuda", dtype=m.torch_dtype)
    ws = torch.empty(kvr.kvr_workspace_bytes(s.handle, 0), dtype=torch.uint8, device="cuda")
    for workspace in (None, ws):
        out.zero_()
        kvr.kvr_attend(s.handle, 0, q, out, workspace, 0 if workspace is None else ws.numel())
        s.sync()
        assert_close(f64(out), want, TOL["bf16"], f"{kind}, workspace={workspace is not None}")
        assert_rel_heads(f64(out), want, TOL["bf16"], m.head_dim, f"{kind}, workspace={workspace is not None}")
    s.close()
