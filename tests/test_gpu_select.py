"""GPU parity of the selection pack: sorted positions, intervals, bit masks,
plan and gathered rows are bit-exact against the oracle's integer
bookkeeping (and host validation rejects malformed supports)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from selective_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

kvr = pytest.importorskip("selective_kv_cache_gb300.kvr")
from selective_kv_cache_gb300.harness import Setup  # noqa: E402
from helpers import small_bf16  # noqa: E402


def one_layer(w):
    """The same workload with a single layer (selection does not depend on depth)."""
    return dataclasses.replace(w, model=dataclasses.replace(w.model, n_layers=1))


def check_selection(s: Setup):
    w = s.w
    local, sink = s.local_mask, s.sink_mask
    off = 0
    for seq, pos in enumerate(s.positions):
        n = len(pos)
        U = oracle.sorted_positions(pos)
        iv = oracle.intervals(U)
        got = kvr.kvr_read_selection(s.handle, seq, n, iv.shape[0], s.words)
        np.testing.assert_array_equal(got["U"], U)
        np.testing.assert_array_equal(got["intervals"], iv)
        selm = np.zeros(w.capacity, bool)
        selm[U] = True
        loc, snk = oracle.effective_masks(local[seq], sink[seq], selm, bool(s.flags & kvr.KVR_SINK_STATIC))
        np.testing.assert_array_equal(got["sel"], oracle.bitmask_words(selm))
        np.testing.assert_array_equal(got["eloc"], oracle.bitmask_words(loc))
        np.testing.assert_array_equal(got["esnk"], oracle.bitmask_words(snk))
        if n:
            plan = oracle.tile_plan(U, got["rows_per_tile"], got["keys_per_tile"])
            np.testing.assert_array_equal(got["plan"], plan)
        # gathered rows: the row source at the sorted positions, bit for bit
        if s.embed is not None:
            ids = s.ids[seq].cpu().numpy()
            want = s.embed.cpu()[torch.from_numpy(ids[U].astype(np.int64))]
        else:
            want = s.hidden_src[seq].cpu()[torch.from_numpy(U)]
        got_rows = s.hidden[off:off + n].cpu()
        assert torch.equal(got_rows.view(torch.int16) if got_rows.dtype == torch.bfloat16 else got_rows,
                           want.view(torch.int16) if want.dtype == torch.bfloat16 else want)
        off += n


@pytest.mark.parametrize("name", ["tiny", "llama8b", "llama8b_frag", "qwen7b_seam", "qwen1p5b_drift"])
def test_select_pack_bit_exact(name):
    w = one_layer(wl.WORKLOADS[name])
    s = Setup(w)
    rows, ivs = s.select()
    s.sync()
    assert rows == sum(len(p) for p in s.positions)
    assert ivs == sum(oracle.intervals(oracle.sorted_positions(p)).shape[0] for p in s.positions)
    check_selection(s)
    if name == "qwen7b_seam":
        assert ivs == 8 and rows == 896
    s.close()


def test_select_sink_static_and_edges():
    w = small_bf16(n_layers=1, selection="isolated", n_select=97, batch=3)
    rng = np.random.default_rng(5)
    local = rng.random((3, w.capacity)) < 0.5
    sink = rng.random((3, w.capacity)) < 0.3
    pos = [np.array([w.n_tokens - 1], np.int32),                       # the last valid row only
           np.array([], np.int32),                                      # an empty sequence
           rng.permutation(np.arange(w.suffix_start, w.n_tokens))[:333].astype(np.int32)]
    s = Setup(w, positions=pos, local=local, sink=sink, flags=kvr.KVR_SINK_STATIC)
    s.select()
    s.sync()
    check_selection(s)
    s.close()


def test_select_rejects_bad_supports():
    w = small_bf16(n_layers=1, n_select=10)
    s = Setup(w, positions=[np.arange(w.suffix_start, w.suffix_start + 10, dtype=np.int32)])
    s.select()
    good = s.pos_host.copy()
    for bad, code in [([w.suffix_start - 1], kvr.KVR_ERANGE), ([w.n_tokens], kvr.KVR_ERANGE),
                      ([w.suffix_start + 3, w.suffix_start + 3], kvr.KVR_EINVAL)]:
        s.pos_host = np.array(bad, np.int32)
        s.counts = np.array([len(bad)], np.int32)
        with pytest.raises(kvr.KvrError) as e:
            s.select()
        assert e.value.status == code
    # exact budget (Eq. 3): S = 800, b = 2 -> 16 positions required
    s.pos_host, s.counts = good, np.array([10], np.int32)
    with pytest.raises(kvr.KvrError) as e:
        s.select(budget_percent=2)
    assert e.value.status == kvr.KVR_EINVAL
    s.pos_host = np.arange(w.suffix_start, w.suffix_start + 16, dtype=np.int32)
    s.counts = np.array([16], np.int32)
    s.positions = [s.pos_host]
    s.select(budget_percent=2)
    s.sync()
    check_selection(s)
    s.close()
