"""ctypes binding of libbpkv (include/bpkv.h): argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
tensors (or raw integer pointers) for the pointer arguments and the current
CUDA stream unless one is given, and raises ``BpkvError`` on a non-zero
status.  All computation happens in the library's CUDA kernels; if the library
is missing this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(_HERE), "include", "bpkv.h")

P = ctypes.c_void_p
i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


class BpkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = _lib.bpkv_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: {msg} ({status})")


class bpkv_cache(ctypes.Structure):
    _fields_ = [
        ("n_seq", i32), ("n_kv_heads", i32), ("group", i32), ("head_dim", i32),
        ("cap_tokens", i64), ("n_max", i64), ("residency", i32), ("reserved", i32),
        ("planes", P), ("scales", P), ("k_rows", P), ("v_rows", P), ("seq_len", P), ("basis", P),
        ("vplanes", P), ("vscales", P), ("rc_rows", P), ("rc_tok", P), ("rc_slots", i32), ("rc_reserved", i32),
    ]


class bpkv_step_args(ctypes.Structure):
    _fields_ = [
        ("k_new", P), ("v_new", P), ("q", P), ("sigma2", P), ("budget_q", P),
        ("depth_rule", i32), ("fixed_channels", i32), ("fixed_depth", i32),
        ("k", i32), ("n_sink", i32), ("n_recent", i32),
        ("out", P), ("depths_out", P), ("idx_out", P), ("stage_events", P), ("flags", i32),
        ("depths_in", P), ("budget_v", i32), ("vdepth_out", P),
    ]


_SIGS = {
    "bpkv_version": ([], i32),
    "bpkv_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "bpkv_workspace_size": ([P, i32, i32], sz),
    "bpkv_clear_status": ([P, P], ctypes.c_int),
    "bpkv_read_status": ([P, P, P], ctypes.c_int),
    "bpkv_selftest_wait": ([P, i32, i32, P], ctypes.c_int),
    "bpkv_row_cache_stats": ([P, i32, P, P, P], ctypes.c_int),
    "bpkv_selection_map": ([P, i32, P, P, P], ctypes.c_int),
    "bpkv_encode_append": ([P, P, P, i32, P], ctypes.c_int),
    "bpkv_alloc_depths": ([P, P, P, P, P, P], ctypes.c_int),
    "bpkv_fixed_depths": ([P, P, i32, i32, P, P], ctypes.c_int),
    "bpkv_calibrate_channels": ([P, P, i32, i32, i64, i64, i32, i32, P, P], ctypes.c_int),
    "bpkv_rotate": ([P, i32, i32, i64, P, P, P], ctypes.c_int),
    "bpkv_scan": ([P, P, P, P, i64, P], ctypes.c_int),
    "bpkv_topk": ([P, P, i64, i32, i32, i32, P, P, sz, P], ctypes.c_int),
    "bpkv_scan_topk": ([P, P, P, i32, i32, i32, P, P, sz, P], ctypes.c_int),
    "bpkv_scan_topk_noalloc": ([P, P, P, i32, i32, i32, P, P], ctypes.c_int),
    "bpkv_union": ([P, P, i32, P, P, P, P], ctypes.c_int),
    "bpkv_sparse_attend": ([P, P, P, P, P, i32, P, P, sz, P], ctypes.c_int),
    "bpkv_dense_attend": ([P, P, P, P, sz, P], ctypes.c_int),
    "bpkv_sparse_attend_vdepth": ([P, P, P, P, P, i32, i32, P, P, P, P], ctypes.c_int),
    "bpkv_decode_step": ([P, i32, P, P, sz, P], ctypes.c_int),
}

_lib = None


def lib_path() -> str:
    from .build import lib_path as _lp
    return _lp()


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libbpkv (built by ``bit_plane_kv_encode_gb300.build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path()
    if not os.path.exists(p):
        raise ImportError(f"libbpkv is not built ({p} missing); run __graft_entry__.build()")
    L = ctypes.CDLL(p)
    for name, (args, res) in _SIGS.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    if path is None:
        _lib = L
    return L


def header_symbols() -> list:
    """Names of the functions declared in include/bpkv.h."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\w[\w\s\*]*?\b(bpkv_\w+)\s*\(", txt, flags=re.M)))


# ------------------------------------------------------------------ marshalling

def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    return ctypes.c_void_p(x.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, rc: int) -> int:
    if rc != 0:
        raise BpkvError(fn, rc)
    return rc


def bpkv_version() -> int:
    return int(load().bpkv_version())


def bpkv_status_string(status: int) -> str:
    return load().bpkv_status_string(int(status)).decode()


def bpkv_workspace_size(cache, k: int, what: int) -> int:
    return int(load().bpkv_workspace_size(ctypes.byref(cache), int(k), int(what)))


def bpkv_clear_status(ws, stream=None):
    return _check("bpkv_clear_status", load().bpkv_clear_status(_ptr(ws), _stream(stream)))


def bpkv_read_status(ws, stream=None) -> int:
    st = ctypes.c_int32(0)
    rc = load().bpkv_read_status(_ptr(ws), ctypes.byref(st), _stream(stream))
    if rc not in (0, -5):
        _check("bpkv_read_status", rc)
    return int(st.value)


def bpkv_row_cache_stats(cache, k: int, ws, stream=None):
    """(hits, misses) per (sequence, KV head) of the last step: numpy uint32 [N][H][2]."""
    import numpy as np
    out = np.zeros((cache.n_seq, cache.n_kv_heads, 2), dtype=np.uint32)
    _check("bpkv_row_cache_stats", load().bpkv_row_cache_stats(ctypes.byref(cache), int(k), _ptr(ws),
                                                                out.ctypes.data_as(ctypes.c_void_p), _stream(stream)))
    return out


def bpkv_selection_map(cache, k: int, ws, stream=None):
    """The last step's selection map of its last layer: numpy uint32 [N][H][G][cap_tokens / 32]."""
    import numpy as np
    out = np.zeros((cache.n_seq, cache.n_kv_heads, cache.group, cache.cap_tokens // 32), dtype=np.uint32)
    _check("bpkv_selection_map", load().bpkv_selection_map(ctypes.byref(cache), int(k), _ptr(ws),
                                                            out.ctypes.data_as(ctypes.c_void_p), _stream(stream)))
    return out


def bpkv_selftest_wait(ws, arrivals: int, spin_limit: int, stream=None):
    return _check("bpkv_selftest_wait", load().bpkv_selftest_wait(_ptr(ws), int(arrivals), int(spin_limit),
                                                                  _stream(stream)))


def bpkv_encode_append(cache, k_new, v_new, t_new: int, stream=None):
    return _check("bpkv_encode_append",
                  load().bpkv_encode_append(ctypes.byref(cache), _ptr(k_new), _ptr(v_new), int(t_new),
                                            _stream(stream)))


def bpkv_alloc_depths(cache, q, sigma2, budget_q, depths, stream=None):
    return _check("bpkv_alloc_depths",
                  load().bpkv_alloc_depths(ctypes.byref(cache), _ptr(q), _ptr(sigma2), _ptr(budget_q),
                                           _ptr(depths), _stream(stream)))


def bpkv_fixed_depths(cache, q, n_channels: int, depth: int, depths, stream=None):
    return _check("bpkv_fixed_depths",
                  load().bpkv_fixed_depths(ctypes.byref(cache), _ptr(q), int(n_channels), int(depth),
                                           _ptr(depths), _stream(stream)))


def bpkv_calibrate_channels(q_cal, k_cal, n_units: int, group: int, m_q: int, m_k: int, n_channels: int,
                            depth: int, depths, stream=None):
    return _check("bpkv_calibrate_channels",
                  load().bpkv_calibrate_channels(_ptr(q_cal), _ptr(k_cal), int(n_units), int(group), int(m_q),
                                                 int(m_k), int(n_channels), int(depth), _ptr(depths),
                                                 _stream(stream)))


def bpkv_rotate(basis, n_seq: int, n_kv_heads: int, rows: int, x, y, stream=None):
    return _check("bpkv_rotate", load().bpkv_rotate(_ptr(basis), int(n_seq), int(n_kv_heads), int(rows), _ptr(x),
                                                    _ptr(y), _stream(stream)))


def bpkv_scan(cache, q, depths, scores, ld_scores: int, stream=None):
    return _check("bpkv_scan", load().bpkv_scan(ctypes.byref(cache), _ptr(q), _ptr(depths), _ptr(scores),
                                                int(ld_scores), _stream(stream)))


def bpkv_topk(cache, scores, ld_scores: int, k: int, n_sink: int, n_recent: int, idx, ws, ws_bytes: int,
              stream=None):
    return _check("bpkv_topk",
                  load().bpkv_topk(ctypes.byref(cache), _ptr(scores), int(ld_scores), int(k), int(n_sink),
                                   int(n_recent), _ptr(idx), _ptr(ws), int(ws_bytes), _stream(stream)))


def bpkv_scan_topk(cache, q, depths, k: int, n_sink: int, n_recent: int, idx, ws, ws_bytes: int, stream=None):
    return _check("bpkv_scan_topk",
                  load().bpkv_scan_topk(ctypes.byref(cache), _ptr(q), _ptr(depths), int(k), int(n_sink),
                                        int(n_recent), _ptr(idx), _ptr(ws), int(ws_bytes), _stream(stream)))


def bpkv_scan_topk_noalloc(cache, q, depths, k: int, n_sink: int, n_recent: int, idx, stream=None):
    return _check("bpkv_scan_topk_noalloc",
                  load().bpkv_scan_topk_noalloc(ctypes.byref(cache), _ptr(q), _ptr(depths), int(k), int(n_sink),
                                                int(n_recent), _ptr(idx), _stream(stream)))


def bpkv_union(cache, idx, k: int, uidx, umask, ucount, stream=None):
    return _check("bpkv_union", load().bpkv_union(ctypes.byref(cache), _ptr(idx), int(k), _ptr(uidx),
                                                  _ptr(umask), _ptr(ucount), _stream(stream)))


def bpkv_sparse_attend(cache, q, uidx, umask, ucount, u_cap: int, out, ws, ws_bytes: int, stream=None):
    return _check("bpkv_sparse_attend",
                  load().bpkv_sparse_attend(ctypes.byref(cache), _ptr(q), _ptr(uidx), _ptr(umask), _ptr(ucount),
                                            int(u_cap), _ptr(out), _ptr(ws), int(ws_bytes), _stream(stream)))


def bpkv_sparse_attend_vdepth(cache, q, uidx, umask, ucount, u_cap: int, budget_v: int, out, vdepth=None,
                              weight=None, stream=None):
    return _check("bpkv_sparse_attend_vdepth",
                  load().bpkv_sparse_attend_vdepth(ctypes.byref(cache), _ptr(q), _ptr(uidx), _ptr(umask), _ptr(ucount),
                                                   int(u_cap), int(budget_v), _ptr(out), _ptr(vdepth), _ptr(weight),
                                                   _stream(stream)))


def bpkv_dense_attend(cache, q, out, ws, ws_bytes: int, stream=None):
    return _check("bpkv_dense_attend",
                  load().bpkv_dense_attend(ctypes.byref(cache), _ptr(q), _ptr(out), _ptr(ws), int(ws_bytes),
                                           _stream(stream)))


def bpkv_decode_step(layers_array, n_layers: int, args, ws, ws_bytes: int, stream=None):
    return _check("bpkv_decode_step",
                  load().bpkv_decode_step(layers_array, int(n_layers), ctypes.byref(args), _ptr(ws),
                                          int(ws_bytes), _stream(stream)))
