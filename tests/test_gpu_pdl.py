"""Dependent launches change when kernels start, never what they compute: the
same refreshes run in child processes with KVR_PDL=0 (every kernel waits for
the whole stream) and with it on (kernels start during their predecessor and
load what no earlier kernel of the call writes before they wait) must give the
same bits.  Covers a two-layer Llama-3-8B refresh (attention split merged by
a merge kernel), a one-layer block-seam refresh (biased attention, merge by
the last CTA) and the adapter-drift layer-range schedule (two reselects inside
the call)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import dataclasses, hashlib, sys
import torch
sys.path.insert(0, ROOT)
from selective_kv_cache_gb300 import workloads as wl
from selective_kv_cache_gb300.harness import Setup
def digest(t):   # the bytes of a cache, as one sha256 (it is too big to save twice)
    return hashlib.sha256(t.contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()
out = {}
for name, layers in (("llama8b", 2), ("qwen7b_seam", 1)):
    base = wl.WORKLOADS[name]
    w = dataclasses.replace(base, model=dataclasses.replace(base.model, n_layers=layers))
    s = Setup(w)
    for _ in range(3):          # repeated: a stale read would show as a difference in some run
        s.select()
        s.refresh()
    s.sync()
    out[name] = (s.hidden[:s.n_rows].cpu(), digest(s.K), digest(s.V))
    s.close()
base = wl.WORKLOADS["qwen1p5b_drift"]
w = dataclasses.replace(base, model=dataclasses.replace(base.model, n_layers=16), batch=2)
s = Setup(w)
m = w.model
g = torch.Generator(device="cuda").manual_seed(3)
boundary = torch.randn((w.batch, w.capacity, m.d_model), device="cuda", generator=g).to(m.torch_dtype)
r0, r1 = w.range_layers
for _ in range(2):
    s.refresh_range(boundary, r0, r1)
s.sync()
out["drift"] = (s.hidden[:s.n_rows].cpu(), digest(s.K), digest(s.V))
torch.save(out, sys.argv[1])
'''.replace("ROOT", repr(ROOT))


def _run(pdl, path):
    env = dict(os.environ, KVR_PDL=pdl)
    r = subprocess.run([sys.executable, "-c", CHILD, path], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    return torch.load(path)


def test_dependent_launch_gives_the_same_bits(tmp_path):
    off = _run("0", str(tmp_path / "off.pt"))
    on = _run("1", str(tmp_path / "on.pt"))
    for name in ("llama8b", "qwen7b_seam", "drift"):
        assert torch.equal(off[name][0], on[name][0]), f"{name} hidden"
        assert off[name][1] == on[name][1], f"{name} K"
        assert off[name][2] == on[name][2], f"{name} V"
        assert torch.isfinite(on[name][0].float()).all()
