"""GPU parity of the layer-range policy (CacheReforge: Bounded Recovery for
Stale KV Caches under Evolving Adapters, Eqs. 8-9 and the anchor updates)
against the oracle, over a sequence of adapter updates: per-layer drift
within 1e-12 relative, ranges and versions exact."""
import numpy as np
import pytest
import torch

import oracle.policy as OP

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("dtype,n_params", [(torch.bfloat16, 1_000_003), (torch.float32, 77_777)])
def test_policy_sequence_matches_oracle(dtype, n_params):
    L = 28
    g = torch.Generator(device="cuda")
    g.manual_seed(91)
    theta = (0.01 * torch.randn(n_params, generator=g, device="cuda")).to(dtype)
    # synthetic calibration split: 200 conditions with windows around layers 8-16
    rng = np.random.default_rng(17)
    restart = rng.integers(6, 12, 200)
    window = rng.integers(0, 8, 200)
    dist = rng.uniform(0.5, 2.0, 200)
    s = kvr.kvr_policy_sensitivity(L, restart, window, dist)
    np.testing.assert_array_equal(s, OP.sensitivity(L, restart, window, dist))
    pol = kvr.kvr_policy_create(L, theta, s)
    ref = OP.Policy(s, f64(theta), L)
    updates = [(0.6, OP.MOD_V, 10), (0.4, OP.MOD_Q, 8), (1.5, OP.MOD_K, 6), (-0.6, OP.MOD_MLP, 11),
               (3.0, OP.MOD_V, 0), (0.05, OP.MOD_K, 3)]
    seen = set()
    for version, (scale, module, layer) in enumerate(updates, start=1):
        step = torch.randn(n_params, generator=g, device="cuda")
        step = (step / step.norm() * abs(scale)).to(dtype)
        theta = (theta.float() + (step.float() if scale > 0 else -step.float())).to(dtype)
        d, q, rng_gpu = kvr.kvr_policy_plan(pol, L, theta, module, layer)
        dw, qw, rng_ref = ref.plan(f64(theta), module, layer)
        np.testing.assert_allclose(d, dw, rtol=1e-12, atol=0)
        # the decisions q >= 1 are taken away from the threshold
        assert np.all(np.abs(qw - 1.0) > 1e-9)
        assert rng_gpu == rng_ref
        seen.add("reuse" if rng_ref[0] == rng_ref[1] else ("full" if rng_ref[1] == L else "bounded"))
        kvr.kvr_policy_commit(pol, theta, *rng_gpu, version)
        ref.commit(f64(theta), *rng_ref, version)
        np.testing.assert_array_equal(kvr.kvr_policy_versions(pol, L), ref.version)
    assert "bounded" in seen and "reuse" in seen
    kvr.kvr_policy_destroy(pol)


def test_policy_validation():
    theta = torch.zeros(100, device="cuda")
    with pytest.raises(kvr.KvrError):
        kvr.kvr_policy_create(4, theta, [1.0, -1.0, 0.0, 0.0])
    pol = kvr.kvr_policy_create(4, theta, [1.0] * 4)
    for module, layer in [(9, 0), (0, 4), (0, -1)]:
        with pytest.raises(kvr.KvrError):
            kvr.kvr_policy_plan(pol, 4, theta, module, layer)
    with pytest.raises(kvr.KvrError):
        kvr.kvr_policy_commit(pol, theta, 3, 2, 1)
    d, q, rng = kvr.kvr_policy_plan(pol, 4, theta, OP.MOD_K, 1)
    np.testing.assert_array_equal(d, 0.0)
    assert rng == (1, 1)
    kvr.kvr_policy_destroy(pol)
