"""Seeded synthetic inputs for the fixed-order fold (no fold arithmetic here).

Both sides of every parity check draw their inputs from this module: the CPU
oracle and the CUDA library each receive the same arrays. The generators are
written in C (``gen.c``) because the gradient-arena workloads hold up to half
a billion values; rows are independent xorshift64 streams, so a multi-row fill
runs one thread per row.

Workload recipes (each rank r is its own stream):

* ``c1_rows(W, n)``       -- memra-engine 0.128.0 tests/tp_ar_gpu.rs ``vecf``
  values in [-1, 1); rank r seeded 11 + 66 r + n, which reproduces the page's
  seeds 11 + n and 77 + n for ranks 0 and 1.
* ``gradient_rows(W, n)`` -- N(0, 1e-3) with 1% of entries scaled by 1e3,
  rank r seeded 1000 + r.
* ``normal_rows(W, n)``   -- N(0, 1), rank r seeded 2000 + r.
* ``stress_rows(W, n)``   -- log-uniform magnitudes 1e-30..1e4 with random
  sign, 1% signed zeros, 0.1% subnormals, and fixed special columns in
  elements 0..15; rank r seeded 3000 + r.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libdetfold_inputs.so")

KIND_VECF, KIND_GRADIENT, KIND_NORMAL, KIND_STRESS = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library beside it (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
             "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.detfold_gen_rows.restype = ctypes.c_int
            lib.detfold_gen_rows.argtypes = [
                ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def fill_rows(kind: int, ptr: int, W: int, n: int, row_stride: int,
              seed0: int, seed_step: int) -> None:
    """Fill W rows of n f32 at host address ``ptr`` (row r at ptr + 4*r*row_stride)."""
    rc = _get().detfold_gen_rows(kind, ctypes.c_void_p(ptr), W, n, row_stride,
                                 seed0 & (2**64 - 1), seed_step & (2**64 - 1), _threads())
    if rc != 0:
        raise ValueError(f"detfold_gen_rows rejected kind={kind} W={W} n={n} stride={row_stride}")


def rows(kind: int, W: int, n: int, seed0: int, seed_step: int) -> np.ndarray:
    """A fresh ``float32[W, n]`` array of ``kind`` rows."""
    out = np.empty((W, max(n, 0)), dtype=np.float32)
    if W > 0 and n > 0:
        fill_rows(kind, out.ctypes.data, W, n, n, seed0, seed_step)
    return out


def vecf(n: int, seed: int) -> np.ndarray:
    """memra-engine 0.128.0 tests/tp_ar_gpu.rs ``vecf(n, seed)``."""
    return rows(KIND_VECF, 1, n, seed, 0)[0]


def c1_seed(r: int, n: int) -> int:
    return 11 + 66 * r + n


def c1_rows(W: int, n: int) -> np.ndarray:
    return rows(KIND_VECF, W, n, 11 + n, 66)


def gradient_rows(W: int, n: int, seed0: int = 1000) -> np.ndarray:
    return rows(KIND_GRADIENT, W, n, seed0, 1)


def normal_rows(W: int, n: int, seed0: int = 2000) -> np.ndarray:
    return rows(KIND_NORMAL, W, n, seed0, 1)


def stress_rows(W: int, n: int, seed0: int = 3000) -> np.ndarray:
    return rows(KIND_STRESS, W, n, seed0, 1)


# Workload kinds by name, with their seed base and seed step per rank.
RECIPES = {
    "vecf": (KIND_VECF, None, 66),
    "gradient": (KIND_GRADIENT, 1000, 1),
    "normal": (KIND_NORMAL, 2000, 1),
    "stress": (KIND_STRESS, 3000, 1),
}


def recipe_seed0(name: str, n: int) -> int:
    kind, base, _ = RECIPES[name]
    return 11 + n if base is None else base


def fill_recipe(name: str, ptr: int, W: int, n: int, row_stride: int) -> None:
    kind, _, step = RECIPES[name]
    fill_rows(kind, ptr, W, n, row_stride, recipe_seed0(name, n), step)


def recipe_rows(name: str, W: int, n: int) -> np.ndarray:
    kind, _, step = RECIPES[name]
    return rows(kind, W, n, recipe_seed0(name, n), step)
