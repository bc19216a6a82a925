"""Build libdetfold.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit compiles in parallel to an object under
``_build/``; the objects link into ``libdetfold.so`` beside this file. No
fast-math: binary32 adds keep round-to-nearest-even and subnormals
(``-ftz=false -prec-div=true -prec-sqrt=true``), and ``-fmad=false`` rules out
any multiply-add contraction.

The measurement probes (``csrc/probes/*.cu``, the latency floors that graphs
of small folds are compared against) link into a library of their own,
``libdetfold_probes.so``, which the fold library's binding never loads.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdetfold.so")
PROBES_CSRC = os.path.join(CSRC, "probes")
PROBES_LIB = os.path.join(PKG, "libdetfold_probes.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-ftz=false",
              "-prec-div=true", "-prec-sqrt=true", "-fmad=false", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdetfold")
    return path


def _inputs() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + [os.path.join(INCLUDE, "detfold.h"), os.path.abspath(__file__)])


def _probe_inputs() -> list[str]:
    return sorted(glob.glob(os.path.join(PROBES_CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + [os.path.join(INCLUDE, "detfold.h"), os.path.join(INCLUDE, "detfold_probes.h"),
                     os.path.abspath(__file__)])


def stale(lib: str = LIB, inputs=None) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in (inputs if inputs is not None else _inputs()))


def build(force: bool = False, defines: dict | None = None, lib: str = LIB,
          build_dir: str = BUILD_DIR, verbose: bool = False) -> str:
    """Compile and link libdetfold.so (and, for the default library path, the
    probes library); returns the fold library's path.

    ``defines`` adds -D macros (launch-shape knobs of csrc/detfold_launch.cuh).
    """
    if lib == LIB and (force or stale(PROBES_LIB, _probe_inputs())):
        _link(sorted(glob.glob(os.path.join(PROBES_CSRC, "*.cu"))), PROBES_LIB,
              os.path.join(build_dir, "probes"), [], verbose)
    if not force and not defines and not stale(lib):
        return lib
    dflags = [f"-D{k}={v}" for k, v in (defines or {}).items()]
    return _link(sorted(glob.glob(os.path.join(CSRC, "*.cu"))), lib, build_dir, dflags, verbose)


def _link(sources: list[str], lib: str, build_dir: str, dflags: list[str], verbose: bool) -> str:
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *dflags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(sources), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True))
