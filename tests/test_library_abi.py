"""libkvr.so builds, loads without a GPU, and exports every entry point that
include/kvr.h declares (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "kvr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvr_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from selective_kv_cache_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for must in ("kvr_create_cache", "kvr_select", "kvr_refresh_layer", "kvr_attend"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_entry_points() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_export(lib):
    from selective_kv_cache_gb300 import kvr
    assert sorted(kvr.EXPORTS) == declared_entry_points()


def test_host_validation_needs_no_gpu(lib):
    from selective_kv_cache_gb300 import kvr
    # a NULL descriptor and bad shapes are rejected before any CUDA call
    out = ctypes.c_void_p()
    st = kvr.lib.kvr_create_cache(None, 1, 16, None, None, 16, 0, None, None, 0.0, 0.0, 0, None, ctypes.byref(out))
    assert st == kvr.KVR_EINVAL
    d = kvr.kvr_model_desc(1, 256, 4, 3, 64, 1024, 1e4, 1e-5, kvr.KVR_F32, 0)   # 4 % 3 != 0
    st = kvr.lib.kvr_create_cache(ctypes.byref(d), 1, 16, 16, 16, 16, 0, None, None, 0.0, 0.0, 0, None,
                                  ctypes.byref(out))
    assert st == kvr.KVR_EINVAL
    assert "malformed" in kvr.kvr_last_error()
    d = kvr.kvr_model_desc(1, 256, 4, 4, 64, 1024, 1e4, 1e-5, kvr.KVR_BF16, 0)    # bf16 needs head_dim 128
    st = kvr.lib.kvr_create_cache(ctypes.byref(d), 1, 16, 16, 16, 16, 0, None, None, 0.0, 0.0, 0, None,
                                  ctypes.byref(out))
    assert st == kvr.KVR_EUNSUPPORTED
    assert kvr.lib.kvr_select(None, None, None, -1, None, None, 0, None, None, None, None, None) == kvr.KVR_EINVAL
    assert kvr.kvr_workspace_bytes(None, 10) == 0
    assert kvr.lib.kvr_shift(None, 0, 1, None) == kvr.KVR_EINVAL
    assert kvr.lib.kvr_splice(None, 0, 0, 1, None, None, 0, 0, None) == kvr.KVR_EINVAL
    assert kvr.lib.kvr_cache_info(None, None, None) == kvr.KVR_EINVAL


def test_policy_host_logic_needs_no_gpu(lib):
    """Eq. S4 and the calibration of Eqs. 6-7 run on the host: the library's
    answers equal the oracle's on random calibration splits."""
    import numpy as np
    import oracle.policy as OP
    from selective_kv_cache_gb300 import kvr
    for m in range(5):
        for s_ in (0, 5, 27):
            assert kvr.kvr_restart_layer(m, s_, 28) == OP.restart_layer(m, s_, 28)
    assert kvr.kvr_restart_layer(7, 0, 28) == -1 and kvr.kvr_restart_layer(0, 28, 28) == -1
    rng = np.random.default_rng(8)
    for _ in range(20):
        L, n = int(rng.integers(1, 30)), int(rng.integers(0, 60))
        r = rng.integers(0, L, n)
        h = rng.integers(0, 10, n)
        d = rng.random(n) * 3
        np.testing.assert_array_equal(kvr.kvr_policy_sensitivity(L, r, h, d), OP.sensitivity(L, r, h, d))
    with pytest.raises(kvr.KvrError):
        kvr.kvr_policy_sensitivity(3, [5], [1], [0.1])
    assert kvr.lib.kvr_policy_plan(None, None, 0, 0, None, None, None, None) == kvr.KVR_EINVAL
