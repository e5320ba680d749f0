"""Failure paths, made without faulting the GPU.

Host-side injection (KVR_FAULT, read at the start of every library call)
makes one step fail: the device allocations of kvr_create_cache, the
position upload of a selection, every kernel launch of a call, or a refresh
layer marking the device error word as a bounded wait does when it gives up.
Each call must return its documented status, the handle must stay usable or
destroyable, and once the fault is cleared the same handle must work again.
The device-side bounded wait itself runs through kvr_wait_check: a wait on a
barrier phase that nothing completes, with a budget of about a millisecond,
must come back as ETIMEOUT from kvr_sync_status and leave the context
usable."""
import os

import numpy as np
import pytest
import torch

from selective_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup  # noqa: E402
from helpers import small_bf16  # noqa: E402


class fault:
    def __init__(self, spec):
        self.spec = spec

    def __enter__(self):
        os.environ["KVR_FAULT"] = self.spec
        return self

    def __exit__(self, *a):
        os.environ.pop("KVR_FAULT", None)


def small():
    return small_bf16(n_layers=1, selection="isolated", n_select=40)


@pytest.mark.parametrize("spec", ["alloc", "alloc:1", "alloc:5", "alloc:14"])
def test_create_reports_enomem_and_frees_what_it_allocated(spec):
    w = small()
    K = torch.zeros((1, 1, 2, w.capacity, 128), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        with fault(spec), pytest.raises(kvr.KvrError) as e:
            kvr.kvr_create_cache(kvr.model_desc(w.model), 1, w.capacity, K, K, w.n_tokens, w.suffix_start)
        assert e.value.status == kvr.KVR_ENOMEM
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (2 << 20)     # nothing left behind
    kvr.kvr_destroy_cache(None)
    h = kvr.kvr_create_cache(kvr.model_desc(w.model), 1, w.capacity, K, K, w.n_tokens, w.suffix_start)
    kvr.kvr_destroy_cache(h)


def test_failed_upload_leaves_no_selection_and_recovers():
    s = Setup(small())
    s.select()
    with fault("upload"), pytest.raises(kvr.KvrError) as e:
        s.select()
    assert e.value.status == kvr.KVR_ECUDA
    with pytest.raises(kvr.KvrError) as e:
        s.refresh()
    assert e.value.status == kvr.KVR_ESTATE          # the half-made selection is not used
    s.select()
    s.refresh()
    s.sync()
    assert torch.isfinite(s.hidden[:s.n_rows].float()).all()
    s.close()


def test_failed_launch_reports_ecuda_and_recovers():
    s = Setup(small())
    s.select()
    with fault("launch"), pytest.raises(kvr.KvrError) as e:
        s.refresh()
    assert e.value.status == kvr.KVR_ECUDA
    assert "launch" in str(e.value).lower() or "projection" in str(e.value) or "norm" in str(e.value)
    s.sync()
    s.select()
    s.refresh()
    s.sync()
    s.close()


def test_timeout_word_surfaces_as_etimeout_once():
    s = Setup(small())
    s.select()
    with fault("timeout"):
        s.refresh()
    with pytest.raises(kvr.KvrError) as e:
        s.sync()
    assert e.value.status == kvr.KVR_ETIMEOUT
    s.sync()                                          # the word was cleared
    s.select()
    s.refresh()
    s.sync()
    s.close()


def test_device_bounded_wait_gives_up_and_reports_etimeout():
    s = Setup(small())
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    kvr.kvr_wait_check(s.handle, 2_000_000)          # about 1 ms of SM cycles
    t1.record()
    with pytest.raises(kvr.KvrError) as e:
        s.sync()
    assert e.value.status == kvr.KVR_ETIMEOUT
    assert t0.elapsed_time(t1) < 1000.0              # it came back on its own, well inside a second
    s.select()                                       # the context is still usable
    s.refresh()
    s.sync()
    with pytest.raises(kvr.KvrError) as e:
        kvr.kvr_wait_check(s.handle, 0)
    assert e.value.status == kvr.KVR_EINVAL
    s.close()
