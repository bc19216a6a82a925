"""ORACLE -- test infrastructure, not part of the product.

A ctypes wrapper around ``oracle.c``, the plain serial CPU statement of the
fixed-order fold (mamba-rs 0.6.2 src/dist/reducer.rs, ``reduce_sum_reference``
and the module doc's sum-then-multiply mean). Only ``tests/``, the smoke
check and the benchmark's CPU-baseline leg may import this package; the CUDA
library never does, and this package imports nothing of the CUDA library.

Every function is pinned in ``tests/test_oracle_pins.py`` against results
that do not come from this code: an exact rational model of IEEE binary32
addition, closed forms, brute force over rank orders, and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle.c (gcc, strict IEEE flags) into liboracle.so beside it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
             "-std=c11", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_fold.argtypes = [_P, ctypes.c_int, _I64, _P]
            lib.oracle_fold.restype = None
            lib.oracle_fold_stacked.argtypes = [_P, ctypes.c_int, _I64, _P]
            lib.oracle_fold_stacked.restype = None
            lib.oracle_mean_scale.argtypes = [ctypes.c_int]
            lib.oracle_mean_scale.restype = ctypes.c_float
            lib.oracle_scale.argtypes = [_P, _I64, ctypes.c_float]
            lib.oracle_scale.restype = None
            lib.oracle_allreduce.argtypes = [_P, ctypes.c_int, _I64, ctypes.c_float]
            lib.oracle_allreduce.restype = None
            lib.oracle_shard_plan.argtypes = [_I64, ctypes.c_int, _P, _P]
            lib.oracle_shard_plan.restype = None
            lib.oracle_staged_allreduce.argtypes = [_P, ctypes.c_int, _I64, ctypes.c_float,
                                                    ctypes.c_int, _P]
            lib.oracle_staged_allreduce.restype = None
            lib.oracle_bit_diffs.argtypes = [_P, _P, _I64]
            lib.oracle_bit_diffs.restype = _I64
            _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle works on float32 arrays, got {a.dtype}")
    return a


def _ptr_table(rows) -> tuple[ctypes.Array, list[np.ndarray]]:
    keep = [np.ascontiguousarray(_f32(r)) for r in rows]
    n = {r.shape[0] for r in keep}
    if len(n) > 1:
        raise ValueError("addend length mismatch")
    tab = (ctypes.c_void_p * len(keep))(*[r.ctypes.data for r in keep])
    return tab, keep


def fold(rows) -> np.ndarray:
    """Ascending-rank fold of W equal-length f32 rows (a list or a [W, len] array)."""
    rows = list(rows)
    if len(rows) < 1:
        raise ValueError("need at least one addend")
    tab, keep = _ptr_table(rows)
    n = keep[0].shape[0]
    out = np.empty(n, dtype=np.float32)
    _get().oracle_fold(tab, len(keep), n, out.ctypes.data)
    return out


def fold_stacked(stacked: np.ndarray) -> np.ndarray:
    """Fold of a row-major [W, len] f32 array, slot = source rank."""
    st = np.ascontiguousarray(_f32(stacked))
    W, n = st.shape
    if W < 1:
        raise ValueError("need at least one addend")
    out = np.empty(n, dtype=np.float32)
    _get().oracle_fold_stacked(st.ctypes.data, W, n, out.ctypes.data)
    return out


def mean_scale(W: int) -> np.float32:
    """fl(1/W) in binary32."""
    return np.float32(_get().oracle_mean_scale(int(W)))


def scale(buf: np.ndarray, s) -> np.ndarray:
    """A new array fl(buf * s) (s == 1.0 leaves the values as they are)."""
    out = np.array(_f32(buf), dtype=np.float32, copy=True, order="C")
    _get().oracle_scale(out.ctypes.data, out.shape[0], float(np.float32(s)))
    return out


def allreduce(arenas: list[np.ndarray], s=1.0) -> None:
    """In place: every arena := fold(all arenas) * s."""
    for a in arenas:
        if not (isinstance(a, np.ndarray) and a.dtype == np.float32 and a.flags.c_contiguous):
            raise TypeError("arenas must be C-contiguous float32 arrays")
    tab, keep = _ptr_table(arenas)
    _get().oracle_allreduce(tab, len(keep), keep[0].shape[0], float(np.float32(s)))


def staged_allreduce(arenas: list[np.ndarray], s=1.0, reverse: bool = False) -> None:
    """In place: the reference's owner-shard dataflow (exchange, fold, distribute)."""
    for a in arenas:
        if not (isinstance(a, np.ndarray) and a.dtype == np.float32 and a.flags.c_contiguous):
            raise TypeError("arenas must be C-contiguous float32 arrays")
    tab, keep = _ptr_table(arenas)
    W, n = len(keep), keep[0].shape[0]
    shard = -(-n // W) if W else 0
    stack = np.empty(max(1, W * shard), dtype=np.float32)
    _get().oracle_staged_allreduce(tab, W, n, float(np.float32(s)), int(bool(reverse)),
                                   stack.ctypes.data)


def shard_plan(length: int, W: int) -> tuple[np.ndarray, np.ndarray]:
    if W < 1:
        raise ValueError("W must be >= 1")
    starts = np.empty(W, dtype=np.int64)
    lens = np.empty(W, dtype=np.int64)
    _get().oracle_shard_plan(int(length), int(W), starts.ctypes.data, lens.ctypes.data)
    return starts, lens


def bit_diffs(a: np.ndarray, b: np.ndarray) -> int:
    a = np.ascontiguousarray(_f32(a))
    b = np.ascontiguousarray(_f32(b))
    if a.shape != b.shape:
        raise ValueError("length mismatch")
    return int(_get().oracle_bit_diffs(a.ctypes.data, b.ctypes.data, a.size))
