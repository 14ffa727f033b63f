"""Python side of the CPU oracle (numpy arrays in, numpy arrays out).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference arm of ``bench.py``.  The product library
never imports it.

Each function handles one unit, i.e. one (sequence, KV head) of one layer, and
wraps the C function of the same name in ``bpkv_oracle.c`` (see that file for
the passages of the Fathom page each one follows; the ``v_*`` functions and
``attend_vdepth`` follow the ReadKV page's second read stage).  ``decode_unit``
chains them in the order of one decode step.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bpkv_oracle.c")
_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return os.path.join(_HERE, f"liboracle_{platform.machine()}.so")


def build(force: bool = False, cflags=None) -> str:
    """Compile the oracle with gcc (plain C11, IEEE arithmetic, no contraction)."""
    tag = hashlib.sha1(" ".join(cflags).encode()).hexdigest()[:12] if cflags is not None else ""
    out = lib_path() if cflags is None else os.path.join(_HERE, f"liboracle_{platform.machine()}_{tag}.so")
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", out, _SRC, "-lm"] + list(cflags or [])
        subprocess.run(cmd, check=True)
    return out


def _bind(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, u16, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint16, ctypes.c_double
    L.or_fp16_bits.argtypes = [f64]
    L.or_fp16_bits.restype = u16
    L.or_fp16_value.argtypes = [u16]
    L.or_fp16_value.restype = f64
    L.or_dequant.argtypes = [f64, ctypes.c_int, ctypes.c_int]
    L.or_dequant.restype = f64
    L.or_encode.argtypes = [i64, i32, P, i64, P, P]
    L.or_encode.restype = None
    L.or_alloc_depths.argtypes = [i32, i32, P, P, i32, P]
    L.or_alloc_depths.restype = i32
    L.or_fixed_depths.argtypes = [i32, i32, P, i32, i32, P]
    L.or_fixed_depths.restype = None
    L.or_calibrate_channels.argtypes = [i32, i32, i64, P, i64, P, i32, i32, P]
    L.or_calibrate_channels.restype = None
    L.or_rotate.argtypes = [i32, i64, P, P, P]
    L.or_rotate.restype = None
    L.or_rotate_keys.argtypes = [i32, i64, P, P, P]
    L.or_rotate_keys.restype = None
    L.or_scores.argtypes = [i64, i32, i32, P, P, i64, P, P, P]
    L.or_scores.restype = None
    L.or_topk.argtypes = [i64, P, i32, i32, i32, P]
    L.or_topk.restype = i32
    L.or_union.argtypes = [i32, i32, P, P, P]
    L.or_union.restype = i32
    L.or_attend.argtypes = [i32, i32, P, P, P, P, i32, P]
    L.or_attend.restype = None
    L.or_dense_attend.argtypes = [i64, i32, i32, P, P, P, P]
    L.or_dense_attend.restype = None
    L.or_v_encode.argtypes = [i64, i32, P, P, P]
    L.or_v_encode.restype = None
    L.or_v_row.argtypes = [i32, P, P, i64, ctypes.c_int, P]
    L.or_v_row.restype = None
    L.or_v_alloc.argtypes = [i32, P, i32, P]
    L.or_v_alloc.restype = i32
    L.or_attend_vdepth.argtypes = [i32, i32, P, P, P, P, P, P, i32, i32, P, P, P, P]
    L.or_attend_vdepth.restype = None
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def load_variant(cflags) -> "Oracle":
    """An oracle compiled with extra flags (used to plant mistakes in tests)."""
    return Oracle(_bind(build(force=True, cflags=cflags)))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """Bound oracle functions (default build unless another library is given)."""

    def __init__(self, L: ctypes.CDLL | None = None):
        self.L = L if L is not None else lib()

    # -- scalars
    def fp16_bits(self, x: float) -> int:
        return int(self.L.or_fp16_bits(float(x)))

    def fp16_value(self, h: int) -> float:
        return float(self.L.or_fp16_value(int(h)))

    def dequant(self, s: float, c_t: int, t: int) -> float:
        return float(self.L.or_dequant(float(s), int(c_t), int(t)))

    # -- one unit
    def encode(self, k_bits: np.ndarray, nb_cap: int):
        """k_bits: bf16 patterns [n][D] -> (scales [D][nb_cap] u16, planes [D][4][nb_cap] u64)."""
        k_bits = _c(k_bits, np.uint16)
        n, D = k_bits.shape
        scales = np.zeros((D, nb_cap), dtype=np.uint16)
        planes = np.zeros((D, 4, nb_cap), dtype=np.uint64)
        self.L.or_encode(n, D, _p(k_bits), nb_cap, _p(scales), _p(planes))
        return scales, planes

    def alloc_depths(self, q: np.ndarray, sigma2: np.ndarray, budget_q: int) -> np.ndarray:
        q = _c(q, np.float32)
        s2 = _c(sigma2, np.float32)
        G, D = q.shape
        depth = np.zeros(D, dtype=np.uint8)
        self.L.or_alloc_depths(D, G, _p(q), _p(s2), int(budget_q), _p(depth))
        return depth

    def fixed_depths(self, q: np.ndarray, r: int, t: int) -> np.ndarray:
        q = _c(q, np.float32)
        G, D = q.shape
        depth = np.zeros(D, dtype=np.uint8)
        self.L.or_fixed_depths(D, G, _p(q), int(r), int(t), _p(depth))
        return depth

    def calibrate_channels(self, q_cal: np.ndarray, k_cal_bits: np.ndarray, c: int, t: int) -> np.ndarray:
        """q_cal float [m_q][G][D], k_cal_bits bf16 patterns [m_k][D] -> depths [D]."""
        q_cal = _c(q_cal, np.float32)
        k_cal_bits = _c(k_cal_bits, np.uint16)
        m_q, G, D = q_cal.shape
        depth = np.zeros(D, dtype=np.uint8)
        self.L.or_calibrate_channels(D, G, m_q, _p(q_cal), k_cal_bits.shape[0], _p(k_cal_bits), int(c), int(t),
                                     _p(depth))
        return depth

    def rotate(self, x: np.ndarray, R: np.ndarray) -> np.ndarray:
        """x float [rows][D] -> x R (float32 fused multiply-add chains)."""
        x = _c(x, np.float32)
        R = _c(R, np.float32)
        rows, D = x.reshape(-1, x.shape[-1]).shape
        y = np.zeros(x.shape, dtype=np.float32)
        self.L.or_rotate(D, rows, _p(x), _p(R), _p(y))
        return y

    def rotate_keys(self, k_bits: np.ndarray, R: np.ndarray) -> np.ndarray:
        """bf16 patterns [n][D] -> bf16 patterns of k R."""
        k_bits = _c(k_bits, np.uint16)
        R = _c(R, np.float32)
        n, D = k_bits.shape
        out = np.zeros((n, D), dtype=np.uint16)
        self.L.or_rotate_keys(D, n, _p(k_bits), _p(R), _p(out))
        return out

    def scores(self, n: int, scales: np.ndarray, planes: np.ndarray, depth: np.ndarray,
               q: np.ndarray) -> np.ndarray:
        scales = _c(scales, np.uint16)
        planes = _c(planes, np.uint64)
        depth = _c(depth, np.uint8)
        q = _c(q, np.float32)
        G, D = q.shape
        nb_cap = scales.shape[1]
        out = np.zeros((G, n), dtype=np.float64)
        self.L.or_scores(n, D, G, _p(scales), _p(planes), nb_cap, _p(depth), _p(q), _p(out))
        return out

    def topk(self, score: np.ndarray, k: int, n_sink: int = 4, n_recent: int = 32) -> np.ndarray:
        score = _c(score, np.float64)
        idx = np.full(k, -1, dtype=np.int32)
        self.L.or_topk(score.shape[0], _p(score), int(k), int(n_sink), int(n_recent), _p(idx))
        return idx

    def union(self, idx: np.ndarray):
        idx = _c(idx, np.int32)
        G, k = idx.shape
        uidx = np.full(G * k, -1, dtype=np.int32)
        umask = np.zeros(G * k, dtype=np.uint8)
        u = self.L.or_union(G, k, _p(idx), _p(uidx), _p(umask))
        return uidx[:u].copy(), umask[:u].copy()

    def attend(self, q: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray, idx: np.ndarray) -> np.ndarray:
        q = _c(q, np.float32)
        k_rows = _c(k_rows, np.uint16)
        v_rows = _c(v_rows, np.uint16)
        idx = _c(idx, np.int32)
        G, D = q.shape
        out = np.zeros((G, D), dtype=np.float64)
        self.L.or_attend(D, G, _p(q), _p(k_rows), _p(v_rows), _p(idx), idx.shape[1], _p(out))
        return out

    def dense_attend(self, q: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray, n: int) -> np.ndarray:
        q = _c(q, np.float32)
        k_rows = _c(k_rows, np.uint16)
        v_rows = _c(v_rows, np.uint16)
        G, D = q.shape
        out = np.zeros((G, D), dtype=np.float64)
        self.L.or_dense_attend(int(n), D, G, _p(q), _p(k_rows), _p(v_rows), _p(out))
        return out

    # -- value-side depth (ReadKV page, sections 5.3-5.4)
    def v_encode(self, v_bits: np.ndarray):
        """v_bits: bf16 patterns [n][D] -> (vscales [n] u16, vplanes [n][4][D/64] u64)."""
        v_bits = _c(v_bits, np.uint16)
        n, D = v_bits.shape
        vscales = np.zeros(n, dtype=np.uint16)
        vplanes = np.zeros((n, 4, D // 64), dtype=np.uint64)
        self.L.or_v_encode(n, D, _p(v_bits), _p(vscales), _p(vplanes))
        return vscales, vplanes

    def v_row(self, vscales: np.ndarray, vplanes: np.ndarray, i: int, t: int) -> np.ndarray:
        """Value row i read to depth t -> float64 [D]."""
        vscales = _c(vscales, np.uint16)
        vplanes = _c(vplanes, np.uint64)
        D = vplanes.shape[2] * 64
        out = np.zeros(D, dtype=np.float64)
        self.L.or_v_row(D, _p(vscales), _p(vplanes), int(i), int(t), _p(out))
        return out

    def v_alloc(self, a: np.ndarray, budget: int):
        """Row weights a [n_rows] (float64), budget in planes -> (depths [n_rows] u8, planes used)."""
        a = _c(a, np.float64)
        depth = np.zeros(a.shape[0], dtype=np.uint8)
        used = self.L.or_v_alloc(a.shape[0], _p(a), int(budget), _p(depth))
        return depth, int(used)

    def attend_vdepth(self, q: np.ndarray, k_rows: np.ndarray, vscales: np.ndarray, vplanes: np.ndarray,
                      uidx: np.ndarray, umask: np.ndarray, budget_v: int, depth_in: np.ndarray | None = None) -> dict:
        """Stage 2 over one KV head's union: weights, value depths (allocated, or
        ``depth_in`` when given), output [G][D]."""
        q = _c(q, np.float32)
        k_rows = _c(k_rows, np.uint16)
        vscales = _c(vscales, np.uint16)
        vplanes = _c(vplanes, np.uint64)
        uidx = _c(uidx, np.int32)
        umask = _c(umask, np.uint8)
        G, D = q.shape
        n_u = uidx.shape[0]
        depth = np.zeros(n_u, dtype=np.uint8)
        weight = np.zeros(n_u, dtype=np.float64)
        out = np.zeros((G, D), dtype=np.float64)
        din = None if depth_in is None else _c(depth_in, np.uint8)
        self.L.or_attend_vdepth(D, G, _p(q), _p(k_rows), _p(vscales), _p(vplanes), _p(uidx), _p(umask), n_u,
                                int(budget_v), None if din is None else _p(din), _p(depth), _p(weight), _p(out))
        return dict(depth=depth, weight=weight, out=out)

    def decode_unit(self, k_bits: np.ndarray, v_bits: np.ndarray, q: np.ndarray, sigma2: np.ndarray,
                    budget_bits: int | None, k: int, n_sink: int = 4, n_recent: int = 32,
                    nb_cap: int | None = None, depth: np.ndarray | None = None,
                    fixed: tuple | None = None, basis: np.ndarray | None = None) -> dict:
        """One decode step of one unit: encode the n rows, allocate depths (or
        take ``depth`` / a ``fixed`` rule), score, select, union, attend.  With
        a ``basis`` R the codes are those of the keys k R and the depths and
        scores use q R (sigma2 is then the variance in that basis); the
        attention uses the original q and rows."""
        n, D = k_bits.shape
        nb_cap = nb_cap if nb_cap is not None else (n + 63) // 64
        kq, qq = k_bits, q
        if basis is not None:
            kq, qq = self.rotate_keys(k_bits, basis), self.rotate(q, basis)
        scales, planes = self.encode(kq, nb_cap)
        if depth is None:
            if fixed is not None:
                depth = self.fixed_depths(qq, fixed[0], fixed[1])
            else:
                depth = self.alloc_depths(qq, sigma2, 4 * int(budget_bits))
        sc = self.scores(n, scales, planes, depth, qq)
        G = q.shape[0]
        idx = np.stack([self.topk(sc[h], k, n_sink, n_recent) for h in range(G)])
        uidx, umask = self.union(idx)
        out = self.attend(q, k_bits, v_bits, idx)
        return dict(scales=scales, planes=planes, depth=depth, scores=sc, idx=idx,
                    uidx=uidx, umask=umask, out=out)


def bf16_bits(t) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 bit patterns (CPU copy)."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
