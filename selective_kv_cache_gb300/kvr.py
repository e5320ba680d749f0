"""Python binding of libkvr (include/kvr.h): argument marshalling only.

Every function has the C entry point's name and order of arguments; torch
tensors are passed by their data pointers, streams by their CUDA handle.
Import fails loudly when libkvr.so has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvr.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m selective_kv_cache_gb300.build` "
        "(or __graft_entry__.build()); the refresh has no CPU fallback")
lib = C.CDLL(LIB_PATH)

KVR_OK, KVR_EINVAL, KVR_ERANGE, KVR_ENOMEM, KVR_ECUDA, KVR_ETIMEOUT, KVR_EDEVICE, KVR_ESTATE, KVR_EUNSUPPORTED = range(9)
STATUS_NAMES = ["OK", "EINVAL", "ERANGE", "ENOMEM", "ECUDA", "ETIMEOUT", "EDEVICE", "ESTATE", "EUNSUPPORTED"]
KVR_F32, KVR_BF16 = 0, 1
KVR_SINK_STATIC = 0x1
KVR_COMMIT_META = 0x1
KVR_SPLICE_LOCAL = 0x1
KVR_SPLICE_SINK = 0x2
KVR_MOD_Q, KVR_MOD_K, KVR_MOD_V, KVR_MOD_O, KVR_MOD_MLP = range(5)
KERNELS = ["select", "gather", "rmsnorm", "gemm_qkv", "epi_qkv", "attention", "gemm_o", "epi_o",
           "gemm_gate_up", "epi_gate_up", "gemm_down", "epi_down", "commit"]
KVR_K_COUNT = len(KERNELS)

EXPORTS = ["kvr_create_cache", "kvr_destroy_cache", "kvr_select", "kvr_workspace_bytes",
           "kvr_refresh_layer", "kvr_refresh", "kvr_attend", "kvr_sync_status", "kvr_last_error",
           "kvr_read_selection", "kvr_read_meta", "kvr_profile_enable", "kvr_profile_read",
           "kvr_refresh_layer_noalloc", "kvr_refresh_interval_wise", "kvr_reselect", "kvr_lora_merge",
           "kvr_shift", "kvr_splice", "kvr_cache_info", "kvr_restart_layer", "kvr_policy_sensitivity",
           "kvr_policy_create", "kvr_policy_destroy", "kvr_policy_plan", "kvr_policy_commit", "kvr_policy_versions",
           "kvr_sur_workspace_bytes", "kvr_sur_select", "kvr_sur_status", "kvr_refresh_range",
           "kvr_wait_check"]


class kvr_model_desc(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32),
                ("rope_theta", C.c_double), ("rms_eps", C.c_float), ("dtype", C.c_int32),
                ("has_qkv_bias", C.c_int32), ("has_qk_norm", C.c_int32)]


class kvr_layer_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w_qkv", "b_qkv", "w_o", "w_gate_up", "w_down", "norm1", "norm2",
                                          "q_norm", "k_norm")]


class KvrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.kvr_last_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES[status] if 0 <= status < 9 else status}: {msg}")


P = C.c_void_p
I32 = C.c_int32
lib.kvr_create_cache.argtypes = [C.POINTER(kvr_model_desc), I32, I32, P, P, I32, I32, P, P, C.c_float, C.c_float,
                                 C.c_uint32, P, C.POINTER(P)]
lib.kvr_destroy_cache.argtypes = [P]
lib.kvr_select.argtypes = [P, P, P, I32, P, P, I32, P, P, P, P, P]
lib.kvr_workspace_bytes.argtypes = [P, I32]
lib.kvr_workspace_bytes.restype = C.c_size_t
lib.kvr_refresh_layer.argtypes = [P, I32, C.POINTER(kvr_layer_weights), P, P, C.c_size_t, C.c_uint32, P]
lib.kvr_refresh_layer_noalloc.argtypes = [P, I32, C.POINTER(kvr_layer_weights), P, C.c_uint32, P]
lib.kvr_refresh_interval_wise.argtypes = [P, P, P, I32, P, P, I32, P, C.POINTER(kvr_layer_weights), I32, I32, P, P,
                                          C.c_size_t, C.c_uint32, P, P]
lib.kvr_reselect.argtypes = [P, P, P, P, P, P, P, P, P]
lib.kvr_refresh_range.argtypes = [P, C.POINTER(kvr_layer_weights), I32, I32, P, P, P, P, I32, P, P, P, P, P,
                                  C.c_size_t, C.c_uint32, P]
lib.kvr_lora_merge.argtypes = [P, P, I32, I32, I32, I32, P, P, I32, C.c_float, I32, P]
lib.kvr_shift.argtypes = [P, I32, I32, P]
lib.kvr_splice.argtypes = [P, I32, I32, I32, P, P, I32, C.c_uint32, P]
lib.kvr_cache_info.argtypes = [P, P, P]
lib.kvr_restart_layer.argtypes = [I32, I32, I32]
lib.kvr_policy_sensitivity.argtypes = [I32, I32, P, P, P, P]
lib.kvr_policy_create.argtypes = [I32, C.c_int64, I32, P, P, P, C.POINTER(P)]
lib.kvr_policy_destroy.argtypes = [P]
lib.kvr_policy_plan.argtypes = [P, P, I32, I32, P, P, P, P]
lib.kvr_policy_commit.argtypes = [P, P, I32, I32, C.c_int64, P]
lib.kvr_policy_versions.argtypes = [P, P]
lib.kvr_sur_workspace_bytes.argtypes = [I32, I32, I32, I32]
lib.kvr_sur_workspace_bytes.restype = C.c_size_t
lib.kvr_sur_select.argtypes = [P, I32, I32, I32, P, I32, I32, P, I32, P, I32, I32, P, C.c_size_t, P, P, P, P]
lib.kvr_sur_status.argtypes = [P, P]
lib.kvr_refresh.argtypes = [P, C.POINTER(kvr_layer_weights), I32, I32, P, P, C.c_size_t, C.c_uint32, P]
lib.kvr_attend.argtypes = [P, I32, P, P, P, C.c_size_t, P]
lib.kvr_sync_status.argtypes = [P, P]
lib.kvr_wait_check.argtypes = [P, C.c_int64, P]
lib.kvr_last_error.restype = C.c_char_p
lib.kvr_restart_layer.restype = C.c_int32
lib.kvr_read_selection.argtypes = [P, I32, P, I32, P, I32, P, P, P, P, I32, P, P, P]
lib.kvr_read_meta.argtypes = [P, P, P]
lib.kvr_profile_enable.argtypes = [P, I32]
lib.kvr_profile_read.argtypes = [P, P, P, I32]
for _f in EXPORTS:
    if _f not in ("kvr_workspace_bytes", "kvr_last_error", "kvr_restart_layer", "kvr_sur_workspace_bytes"):
        getattr(lib, _f).restype = C.c_int


def _check(status: int, where: str):
    if status != KVR_OK:
        raise KvrError(status, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def model_desc(shape) -> kvr_model_desc:
    """kvr_model_desc from any object with the shape attributes."""
    return kvr_model_desc(shape.n_layers, shape.d_model, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                          shape.ffn_dim, float(shape.rope_theta), float(shape.rms_eps),
                          KVR_BF16 if shape.dtype == "bf16" else KVR_F32, int(bool(shape.qkv_bias)),
                          int(bool(getattr(shape, "qk_norm", False))))


def layer_weights(L) -> kvr_layer_weights:
    """kvr_layer_weights from a dict of device tensors (keys as the struct)."""
    return kvr_layer_weights(*[_ptr(L.get(k)) for k in ("w_qkv", "b_qkv", "w_o", "w_gate_up", "w_down",
                                                         "norm1", "norm2", "q_norm", "k_norm")])


def layer_weights_array(layers: Sequence[dict]):
    arr = (kvr_layer_weights * len(layers))()
    for i, L in enumerate(layers):
        arr[i] = layer_weights(L)
    return arr


def kvr_create_cache(desc: kvr_model_desc, batch: int, capacity: int, k_base, v_base, n_tokens: int,
                     suffix_start: int, local_bits=None, sink_bits=None, alpha: float = 0.0, beta: float = 0.0,
                     flags: int = 0, stream=None) -> int:
    """Returns the cache handle (an int).  local_bits / sink_bits: uint32 numpy
    arrays [batch, ceil(capacity/32)] (host) or None."""
    out = P()
    lb = None if local_bits is None else local_bits.ctypes.data
    sb = None if sink_bits is None else sink_bits.ctypes.data
    _check(lib.kvr_create_cache(C.byref(desc), batch, capacity, _ptr(k_base), _ptr(v_base), n_tokens, suffix_start,
                                lb, sb, alpha, beta, flags, _stream(stream), C.byref(out)), "kvr_create_cache")
    return out.value


def kvr_destroy_cache(c: int):
    _check(lib.kvr_destroy_cache(c), "kvr_destroy_cache")


def kvr_select(c: int, positions, counts, budget_percent: int = -1, token_ids=None, embed_table=None,
               vocab: int = 0, hidden_src=None, hidden_out=None, stream=None):
    """positions, counts: host int32 numpy arrays (or pinned int32 tensors).
    Returns (n_rows, n_intervals)."""
    n_rows = I32()
    n_iv = I32()
    pp = positions.ctypes.data if hasattr(positions, "ctypes") else _ptr(positions)
    cp = counts.ctypes.data if hasattr(counts, "ctypes") else _ptr(counts)
    _check(lib.kvr_select(c, pp, cp, budget_percent, _ptr(token_ids), _ptr(embed_table), vocab, _ptr(hidden_src),
                          _ptr(hidden_out), C.byref(n_rows), C.byref(n_iv), _stream(stream)), "kvr_select")
    return n_rows.value, n_iv.value


def kvr_workspace_bytes(c: int, max_rows: int = 0) -> int:
    return lib.kvr_workspace_bytes(c, max_rows)


def kvr_refresh_layer(c: int, layer: int, weights: kvr_layer_weights, hidden_inout, workspace, ws_bytes: int,
                      flags: int = 0, stream=None):
    _check(lib.kvr_refresh_layer(c, layer, C.byref(weights), _ptr(hidden_inout), _ptr(workspace), ws_bytes, flags,
                                 _stream(stream)), "kvr_refresh_layer")


def kvr_refresh_layer_noalloc(c: int, layer: int, weights: kvr_layer_weights, hidden_inout, flags: int = 0,
                              stream=None):
    """kvr_refresh_layer with the library's fixed 64 MiB device scratch instead of
    a caller workspace (nothing is allocated)."""
    _check(lib.kvr_refresh_layer_noalloc(c, layer, C.byref(weights), _ptr(hidden_inout), flags, _stream(stream)),
           "kvr_refresh_layer_noalloc")


def kvr_refresh(c: int, weights_array, layer_begin: int, layer_end: int, hidden_inout, workspace, ws_bytes: int,
                flags: int = 0, stream=None):
    _check(lib.kvr_refresh(c, weights_array, layer_begin, layer_end, _ptr(hidden_inout), _ptr(workspace), ws_bytes,
                           flags, _stream(stream)), "kvr_refresh")


def kvr_refresh_interval_wise(c: int, positions, counts, budget_percent: int = -1, token_ids=None, embed_table=None,
                              vocab: int = 0, hidden_src=None, weights_array=None, layer_begin: int = 0,
                              layer_end: int = 0, hidden_out=None, workspace=None, ws_bytes: int = 0,
                              flags: int = KVR_COMMIT_META, stream=None) -> int:
    """Returns the number of intervals."""
    n_iv = I32()
    pp = positions.ctypes.data if hasattr(positions, "ctypes") else _ptr(positions)
    cp = counts.ctypes.data if hasattr(counts, "ctypes") else _ptr(counts)
    _check(lib.kvr_refresh_interval_wise(c, pp, cp, budget_percent, _ptr(token_ids), _ptr(embed_table), vocab,
                                         _ptr(hidden_src), weights_array, layer_begin, layer_end, _ptr(hidden_out),
                                         _ptr(workspace), ws_bytes, flags, C.byref(n_iv), _stream(stream)),
           "kvr_refresh_interval_wise")
    return n_iv.value


def kvr_reselect(c: int, positions, counts, carry_rows, fill_rows, hidden_out, stream=None):
    n_rows = I32()
    n_iv = I32()
    pp = positions.ctypes.data if hasattr(positions, "ctypes") else _ptr(positions)
    cp = counts.ctypes.data if hasattr(counts, "ctypes") else _ptr(counts)
    _check(lib.kvr_reselect(c, pp, cp, _ptr(carry_rows), _ptr(fill_rows), _ptr(hidden_out), C.byref(n_rows),
                            C.byref(n_iv), _stream(stream)), "kvr_reselect")
    return n_rows.value, n_iv.value


def kvr_refresh_range(c: int, weights_array, range_begin: int, range_end: int, positions, counts, token_ids=None,
                      embed_table=None, vocab: int = 0, hidden_src=None, boundary=None, hidden_sel=None,
                      hidden_full=None, workspace=None, ws_bytes: int = 0, flags: int = KVR_COMMIT_META, stream=None):
    pp = positions.ctypes.data if hasattr(positions, "ctypes") else _ptr(positions)
    cp = counts.ctypes.data if hasattr(counts, "ctypes") else _ptr(counts)
    _check(lib.kvr_refresh_range(c, weights_array, range_begin, range_end, pp, cp, _ptr(token_ids),
                                 _ptr(embed_table), vocab, _ptr(hidden_src), _ptr(boundary), _ptr(hidden_sel),
                                 _ptr(hidden_full), _ptr(workspace), ws_bytes, flags, _stream(stream)),
           "kvr_refresh_range")


def kvr_wait_check(c: int, cycles: int, stream=None):
    _check(lib.kvr_wait_check(c, cycles, _stream(stream)), "kvr_wait_check")


def kvr_lora_merge(w, w_out, n_out: int, K: int, row_begin: int, row_count: int, a, b, rank: int, scale: float,
                   dtype: int, stream=None):
    _check(lib.kvr_lora_merge(_ptr(w), _ptr(w_out), n_out, K, row_begin, row_count, _ptr(a), _ptr(b), rank, scale,
                              dtype, _stream(stream)), "kvr_lora_merge")


def kvr_shift(c: int, start: int, d: int, stream=None):
    _check(lib.kvr_shift(c, start, d, _stream(stream)), "kvr_shift")


def kvr_splice(c: int, seq: int, dst_pos: int, n: int, k_src, v_src, src_pos: int = 0, flags: int = 0,
               stream=None):
    _check(lib.kvr_splice(c, seq, dst_pos, n, _ptr(k_src), _ptr(v_src), src_pos, flags, _stream(stream)),
           "kvr_splice")


def kvr_cache_info(c: int):
    """(n_tokens, suffix_start) of the cache now."""
    n = C.c_int32()
    s = C.c_int32()
    _check(lib.kvr_cache_info(c, C.byref(n), C.byref(s)), "kvr_cache_info")
    return n.value, s.value


def kvr_attend(c: int, layer: int, q, out, workspace=None, ws_bytes: int = 0, stream=None):
    _check(lib.kvr_attend(c, layer, _ptr(q), _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)), "kvr_attend")


def kvr_sync_status(c: int, stream=None):
    _check(lib.kvr_sync_status(c, _stream(stream)), "kvr_sync_status")


def kvr_last_error() -> str:
    return lib.kvr_last_error().decode()


def kvr_read_selection(c: int, seq: int, count: int, n_intervals: int, words: int, max_tiles: int = 4096):
    """Host copies of the device-built selection of sequence `seq`."""
    import numpy as np
    U = np.zeros(max(count, 1), np.int32)
    iv = np.zeros((max(n_intervals, 1), 2), np.int32)
    sel = np.zeros(words, np.uint32)
    eloc = np.zeros(words, np.uint32)
    esnk = np.zeros(words, np.uint32)
    plan = np.zeros((max_tiles, 6), np.int32)
    nt, rpt, kpt = I32(), I32(), I32()
    _check(lib.kvr_read_selection(c, seq, U.ctypes.data, count, iv.ctypes.data, n_intervals, sel.ctypes.data,
                                  eloc.ctypes.data, esnk.ctypes.data, plan.ctypes.data, max_tiles, C.byref(nt),
                                  C.byref(rpt), C.byref(kpt)), "kvr_read_selection")
    return dict(U=U[:count], intervals=iv[:n_intervals], sel=sel, eloc=eloc, esnk=esnk, plan=plan[:nt.value],
                rows_per_tile=rpt.value, keys_per_tile=kpt.value)


def kvr_read_meta(c: int, batch: int, words: int):
    import numpy as np
    local = np.zeros((batch, words), np.uint32)
    sink = np.zeros((batch, words), np.uint32)
    _check(lib.kvr_read_meta(c, local.ctypes.data, sink.ctypes.data), "kvr_read_meta")
    return local, sink


def kvr_profile_enable(c: int, enable: bool = True):
    _check(lib.kvr_profile_enable(c, int(enable)), "kvr_profile_enable")


def kvr_profile_read(c: int):
    """{kernel name: (launches, total ms)} since the last read."""
    ms = (C.c_double * KVR_K_COUNT)()
    n = (C.c_int64 * KVR_K_COUNT)()
    _check(lib.kvr_profile_read(c, ms, n, KVR_K_COUNT), "kvr_profile_read")
    return {KERNELS[i]: (int(n[i]), float(ms[i])) for i in range(KVR_K_COUNT)}

# ---------------------------------------------------------------- layer-range policy
def kvr_restart_layer(module: int, s: int, n_layers: int) -> int:
    return int(lib.kvr_restart_layer(module, s, n_layers))


def kvr_policy_sensitivity(n_layers: int, restart, window, drift):
    import numpy as np
    r = np.ascontiguousarray(restart, dtype=np.int32)
    w = np.ascontiguousarray(window, dtype=np.int32)
    d = np.ascontiguousarray(drift, dtype=np.float64)
    out = np.zeros(n_layers, np.float64)
    _check(lib.kvr_policy_sensitivity(n_layers, len(r), r.ctypes.data, w.ctypes.data, d.ctypes.data,
                                      out.ctypes.data), "kvr_policy_sensitivity")
    return out


def kvr_policy_create(n_layers: int, theta0, sensitivity, stream=None) -> int:
    """theta0: flat device tensor (bf16 or fp32); sensitivity: n_layers floats."""
    import numpy as np
    s = np.ascontiguousarray(sensitivity, dtype=np.float64)
    out = P()
    dt = KVR_BF16 if theta0.dtype == torch.bfloat16 else KVR_F32
    _check(lib.kvr_policy_create(n_layers, theta0.numel(), dt, _ptr(theta0), s.ctypes.data, _stream(stream),
                                 C.byref(out)), "kvr_policy_create")
    return out.value


def kvr_policy_destroy(p: int):
    _check(lib.kvr_policy_destroy(p), "kvr_policy_destroy")


def kvr_policy_plan(p: int, n_layers: int, theta_t, module: int, update_layer: int, stream=None):
    """Returns (drift [n_layers], risk [n_layers], (begin, end))."""
    import numpy as np
    d = np.zeros(n_layers, np.float64)
    q = np.zeros(n_layers, np.float64)
    rng = np.zeros(2, np.int32)
    _check(lib.kvr_policy_plan(p, _ptr(theta_t), module, update_layer, d.ctypes.data, q.ctypes.data,
                               rng.ctypes.data, _stream(stream)), "kvr_policy_plan")
    return d, q, (int(rng[0]), int(rng[1]))


def kvr_policy_commit(p: int, theta_t, begin: int, end: int, version: int, stream=None):
    _check(lib.kvr_policy_commit(p, _ptr(theta_t), begin, end, version, _stream(stream)), "kvr_policy_commit")


def kvr_policy_versions(p: int, n_layers: int):
    import numpy as np
    v = np.zeros(n_layers, np.int64)
    _check(lib.kvr_policy_versions(p, v.ctypes.data), "kvr_policy_versions")
    return v


# ---------------------------------------------------------------- Semantic-Unit Refresh selection
def kvr_sur_workspace_bytes(S: int, Q: int, d: int, n_units: int) -> int:
    return int(lib.kvr_sur_workspace_bytes(S, Q, d, n_units))


def kvr_sur_select(embed, suffix_ids, query_ids, unit_bounds, budget_percent: int, suffix_start: int, workspace,
                   positions_out, scores_out=None, stream=None) -> int:
    """Device tensors: embed [vocab, d], suffix_ids [S], query_ids [Q],
    unit_bounds [n_units + 1] (int32), workspace (uint8), positions_out int32
    (room for the allowance).  Returns B, the number of positions written."""
    n = I32()
    dt = KVR_BF16 if embed.dtype == torch.bfloat16 else KVR_F32
    _check(lib.kvr_sur_select(_ptr(embed), embed.shape[0], embed.shape[1], dt, _ptr(suffix_ids), suffix_ids.numel(),
                              suffix_start, _ptr(query_ids), query_ids.numel(), _ptr(unit_bounds),
                              unit_bounds.numel() - 1, budget_percent, _ptr(workspace), workspace.numel(),
                              _ptr(positions_out), C.byref(n), _ptr(scores_out), _stream(stream)), "kvr_sur_select")
    return n.value


def kvr_sur_status(workspace, stream=None):
    _check(lib.kvr_sur_status(_ptr(workspace), _stream(stream)), "kvr_sur_status")
