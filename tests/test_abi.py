"""The C-ABI boundary on the CPU: the library loads, exports every declared
symbol, and its host logic (argument validation, the shard plan, status
strings) behaves as include/detfold.h states. No call here reaches a kernel
launch, except the no-device check, which only runs where no GPU exists.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "detfold.h")


@pytest.fixture(scope="module")
def df():
    import deterministic_fixed_order_gb300 as m
    return m


PROBES_HEADER = os.path.join(ROOT, "include", "detfold_probes.h")
PROBES_LIB = os.path.join(ROOT, "deterministic_fixed_order_gb300", "libdetfold_probes.so")

# The fold library's exported API, pinned: the hot-path calls of the boundary,
# the next rows (movement, device tables, one-shot), the allocation-free
# staged call and the plumbing. A symbol added or removed must show up here.
EXPORTED_API = {
    "detfold_sum_stacked", "detfold_sum_ptrs", "detfold_scale", "detfold_loopback_allreduce",
    "detfold_mean_scale", "detfold_staged_workspace_bytes", "detfold_loopback_allreduce_staged",
    "detfold_loopback_allreduce_staged_ex", "detfold_shard_plan", "detfold_status_string",
    "detfold_broadcast", "detfold_all_gather", "detfold_sum_ptrs_dev", "detfold_loopback_allreduce_dev",
    "detfold_one_shot_allreduce", "detfold_loopback_allreduce_staged_noalloc",
    "detfold_last_cuda_error", "detfold_pipeline_timeouts",
}
PROBES_API = {"detfold_probe_launch_floor", "detfold_probe_memory_floor",
              "detfold_probe_same_shape_floor", "detfold_probe_last_cuda_error"}


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(detfold_\w+)\s*\(", text)))


def declaration(name, header=HEADER):
    """The parameter list of one declared function, as (type, name) pairs."""
    text = re.sub(r"/\*.*?\*/", "", open(header).read(), flags=re.S)
    m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
    assert m, name
    params = []
    for p in m.group(1).split(","):
        p = " ".join(p.split())
        if p == "void":
            continue
        typ, nm = re.match(r"(.*?)\s*(\w+)$", p).groups()
        params.append((typ.replace(" *", "*").replace("* ", "*"), nm))
    return params


def test_header_declares_the_api():
    assert set(declared_functions()) == EXPORTED_API
    assert set(declared_functions(PROBES_HEADER)) == PROBES_API


def test_boundary_signatures_are_pinned():
    # the hot-path calls of the boundary and their argument order:
    # (out, inputs, W, len, ..., stream)
    assert declaration("detfold_sum_stacked") == [
        ("float*", "out"), ("const float*", "stacked"), ("int", "W"), ("int64_t", "len"), ("void*", "stream")]
    assert declaration("detfold_sum_ptrs") == [
        ("float*", "out"), ("const float*const*", "srcs"), ("int", "W"), ("int64_t", "len"),
        ("void*", "stream")]
    assert declaration("detfold_scale") == [
        ("float*", "buf"), ("int64_t", "len"), ("float", "scale"), ("void*", "stream")]
    assert declaration("detfold_loopback_allreduce") == [
        ("float*const*", "arenas"), ("int", "W"), ("int64_t", "len"), ("float", "mean_scale"),
        ("void*", "stream")]
    assert declaration("detfold_staged_workspace_bytes") == [("int64_t", "len"), ("int", "W")]
    assert declaration("detfold_loopback_allreduce_staged") == [
        ("float*const*", "arenas"), ("int", "W"), ("int64_t", "len"), ("float", "mean_scale"),
        ("void*", "workspace"), ("int64_t", "workspace_bytes"), ("void*", "stream")]
    assert declaration("detfold_shard_plan") == [
        ("int64_t", "len"), ("int", "W"), ("int64_t*", "starts"), ("int64_t*", "lens")]
    assert declaration("detfold_status_string") == [("int", "status")]
    assert declaration("detfold_mean_scale") == [("int", "W"), ("float*", "scale")]


def test_mean_scale_is_the_binary32_reciprocal(df):
    # fl(1/W), bit for bit the oracle's (itself pinned against the exact
    # rounding model), for every legal W; the binding passes it through
    for W in range(1, 257):
        got = np.float32(df.detfold_mean_scale(W))
        assert got.view(np.uint32) == np.float32(oracle.mean_scale(W)).view(np.uint32), W
        assert df.mean_scale(W) == float(got)
    out = ctypes.c_float(0.0)
    assert df.lib.detfold_mean_scale(0, ctypes.byref(out)) == df.STATUS["DETFOLD_ERR_WORLD"]
    assert df.lib.detfold_mean_scale(257, ctypes.byref(out)) == df.STATUS["DETFOLD_ERR_WORLD"]
    assert df.lib.detfold_mean_scale(4, None) == df.STATUS["DETFOLD_ERR_NULL"]


def test_binding_does_no_method_arithmetic():
    # the binding marshals arguments: no numerics library, no float math
    src = open(os.path.join(ROOT, "deterministic_fixed_order_gb300", "__init__.py")).read()
    assert not re.search(r"^\s*(import numpy|from numpy|import math|from math)", src, re.M)
    assert "float32(" not in src and "1.0 /" not in src and "1 /" not in src


def test_binding_constants_match_the_header(df):
    text = HEADER.read_text() if hasattr(HEADER, "read_text") else open(HEADER).read()
    defs = dict(re.findall(r"^#define (DETFOLD_\w+) (.+)$", text, re.M))

    import ast
    import operator
    ops = {ast.Add: operator.add, ast.Sub: operator.sub, ast.Mult: operator.mul,
           ast.LShift: operator.lshift, ast.USub: operator.neg}

    def arith(node):  # integer constants, + - * << and unary minus only
        if isinstance(node, ast.Constant) and isinstance(node.value, int):
            return node.value
        if isinstance(node, ast.BinOp) and type(node.op) in ops:
            return ops[type(node.op)](arith(node.left), arith(node.right))
        if isinstance(node, ast.UnaryOp) and type(node.op) in ops:
            return ops[type(node.op)](arith(node.operand))
        raise ValueError(f"unexpected header expression: {ast.dump(node)}")

    def value(name):
        expr = re.sub(r"/\*.*", "", defs[name]).strip()
        expr = expr.replace("(int64_t)", "")
        expr = re.sub(r"\b(DETFOLD_\w+)\b", lambda m: f"({value(m.group(1))})", expr)
        return arith(ast.parse(expr, mode="eval").body)

    for name in ("DETFOLD_MAX_W", "DETFOLD_MAX_LEN", "DETFOLD_STAGED_REVERSE_DELIVERY",
                 "DETFOLD_STAGED_SEPARATE_SCALE", "DETFOLD_STAGED_CE_COPIES",
                 "DETFOLD_NOALLOC_SCRATCH_BYTES", "DETFOLD_ONESHOT_MAX_W", "DETFOLD_ONESHOT_MAX_LEN",
                 "DETFOLD_ONESHOT_MAX_CTAS", "DETFOLD_ONESHOT_LINK_BYTES",
                 "DETFOLD_ONESHOT_REFUSE_ENTRY", "DETFOLD_ONESHOT_REFUSE_EXIT"):
        assert getattr(df, name) == value(name), name
    for name, v in df.STATUS.items():
        assert value(name) == v, name


def test_library_exports_only_the_declared_api(df):
    # built with hidden visibility: the dynamic symbol table holds the
    # header's entry points and nothing else of the library
    out = subprocess.run(["nm", "-D", "--defined-only", df.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    defined = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert defined == set(declared_functions()) == EXPORTED_API, sorted(defined ^ EXPORTED_API)


def test_probes_library_exports_only_its_header():
    out = subprocess.run(["nm", "-D", "--defined-only", PROBES_LIB], capture_output=True,
                         text=True, check=True).stdout
    defined = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert defined == PROBES_API, sorted(defined ^ PROBES_API)


def test_library_exports_every_declared_symbol(df):
    out = subprocess.run(["nm", "-D", "--defined-only", df.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (detfold_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        getattr(df.lib, n)  # resolvable through ctypes


def test_header_compiles_as_c():
    src = '#include "detfold.h"\n#include "detfold_probes.h"\nint main(void){return DETFOLD_OK;}\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                        "-x", "c", "-", "-o", os.devnull], input=src, text=True,
                       capture_output=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(df):
    for name, code in df.STATUS.items():
        s = df.detfold_status_string(code)
        assert s and s != "unknown status", name
    assert df.detfold_status_string(12345) == "unknown status"


def test_shard_plan_matches_oracle(df):
    for W in range(1, 12):
        for n in list(range(0, 40)) + [1000003, 100_000_000, (1 << 20) + 7]:
            s, l = df.detfold_shard_plan(n, W)
            os_, ol = oracle.shard_plan(n, W)
            assert s == list(os_) and l == list(ol)


def test_shard_plan_errors(df):
    L = df.lib
    buf = (ctypes.c_int64 * 4)()
    assert L.detfold_shard_plan(10, 0, buf, buf) == df.STATUS["DETFOLD_ERR_WORLD"]
    assert L.detfold_shard_plan(10, 257, buf, buf) == df.STATUS["DETFOLD_ERR_WORLD"]
    assert L.detfold_shard_plan(-1, 4, buf, buf) == df.STATUS["DETFOLD_ERR_LEN"]
    assert L.detfold_shard_plan(10, 4, None, buf) == df.STATUS["DETFOLD_ERR_NULL"]


def test_workspace_bytes(df):
    for n, W in ((100_000_000, 4), ((1 << 20) + 7, 3), (5, 8), (0, 2)):
        b = df.detfold_staged_workspace_bytes(n, W)
        shard = -(-n // W)
        assert b >= W * (shard + 8) * 4 and b % 4 == 0
    assert df.lib.detfold_staged_workspace_bytes(10, 0) == df.STATUS["DETFOLD_ERR_WORLD"]
    assert df.lib.detfold_staged_workspace_bytes(-3, 2) == df.STATUS["DETFOLD_ERR_LEN"]


# Fake device addresses: validation rejects these calls before any launch.
# They are passed only where no GPU exists, so that a validation gap can
# never turn into a launch on addresses that are not device memory.
A = 1 << 32


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available() or os.path.exists("/dev/nvidia0")
    except Exception:
        return True  # unknown: assume a GPU


no_gpu_only = pytest.mark.skipif(_has_gpu(), reason="fake device addresses only where no GPU exists")


def _tab(*ptrs):
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


@no_gpu_only
def test_validation_sum_stacked(df):
    L, S = df.lib, df.STATUS
    assert L.detfold_sum_stacked(None, A, 2, 8, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_sum_stacked(A, None, 2, 8, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_sum_stacked(A, A + 4096, 0, 8, None) == S["DETFOLD_ERR_WORLD"]
    assert L.detfold_sum_stacked(A, A + 4096, 257, 8, None) == S["DETFOLD_ERR_WORLD"]
    assert L.detfold_sum_stacked(A, A + 4096, 2, -1, None) == S["DETFOLD_ERR_LEN"]
    assert L.detfold_sum_stacked(A, A + 4096, 2, (1 << 40) + 1, None) == S["DETFOLD_ERR_LEN"]
    assert L.detfold_sum_stacked(A + 2, A + 4096, 2, 8, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_sum_stacked(A, A + 4098, 2, 8, None) == S["DETFOLD_ERR_ALIGN"]
    # out inside the stacked rows, or overlapping their start
    assert L.detfold_sum_stacked(A + 32, A, 2, 8, None) == S["DETFOLD_ERR_OVERLAP"]
    assert L.detfold_sum_stacked(A, A + 28, 2, 8, None) == S["DETFOLD_ERR_OVERLAP"]
    # len == 0: a no-op once pointers and W are valid
    assert L.detfold_sum_stacked(A, A, 2, 0, None) == S["DETFOLD_OK"]


@no_gpu_only
def test_validation_sum_ptrs(df):
    L, S = df.lib, df.STATUS
    assert L.detfold_sum_ptrs(A, None, 2, 8, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_sum_ptrs(A, _tab(A + 4096, 0), 2, 8, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_sum_ptrs(A, _tab(A + 4096, A + 8192), 0, 8, None) == S["DETFOLD_ERR_WORLD"]
    assert L.detfold_sum_ptrs(A, _tab(A + 4096, A + 8194), 2, 8, None) == S["DETFOLD_ERR_ALIGN"]
    # out partially overlapping a source is refused; out == a source is the in-place fold
    assert L.detfold_sum_ptrs(A, _tab(A + 4, A + 8192), 2, 8, None) == S["DETFOLD_ERR_OVERLAP"]
    assert L.detfold_sum_ptrs(A, _tab(A, A + 8192), 2, 0, None) == S["DETFOLD_OK"]
    # W == 1 in place: nothing to do, nothing launched
    assert L.detfold_sum_ptrs(A, _tab(A), 1, 8, None) == S["DETFOLD_OK"]


@no_gpu_only
def test_validation_allreduce(df):
    L, S = df.lib, df.STATUS
    assert L.detfold_loopback_allreduce(None, 2, 8, 1.0, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_loopback_allreduce(_tab(A, 0), 2, 8, 1.0, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_loopback_allreduce(_tab(A, A + 4096), 300, 8, 1.0, None) == S["DETFOLD_ERR_WORLD"]
    assert L.detfold_loopback_allreduce(_tab(A, A + 4097), 2, 8, 1.0, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_loopback_allreduce(_tab(A, A), 2, 8, 1.0, None) == S["DETFOLD_ERR_OVERLAP"]
    assert L.detfold_loopback_allreduce(_tab(A, A + 16), 2, 8, 1.0, None) == S["DETFOLD_ERR_OVERLAP"]
    assert L.detfold_loopback_allreduce(_tab(A, A + 4096), 2, 0, 0.5, None) == S["DETFOLD_OK"]
    # one rank, scale 1: nothing to do
    assert L.detfold_loopback_allreduce(_tab(A), 1, 8, 1.0, None) == S["DETFOLD_OK"]


@no_gpu_only
def test_validation_staged(df):
    L, S = df.lib, df.STATUS
    ws_need = df.detfold_staged_workspace_bytes(64, 2)
    arenas = _tab(A, A + 4096)
    W_ = A + (1 << 20)
    X = L.detfold_loopback_allreduce_staged_ex
    assert X(arenas, 2, 64, 1.0, 8, W_, ws_need, None) == S["DETFOLD_ERR_ARG"]
    assert X(arenas, 2, 64, 1.0, -1, W_, ws_need, None) == S["DETFOLD_ERR_ARG"]
    for call in (lambda *a: L.detfold_loopback_allreduce_staged(*a[:4], *a[5:]), X):
        assert call(arenas, 2, 64, 1.0, 0, None, ws_need, None) == S["DETFOLD_ERR_WORKSPACE"]
        assert call(arenas, 2, 64, 1.0, 0, W_, ws_need - 4, None) == S["DETFOLD_ERR_WORKSPACE"]
        assert call(arenas, 2, 64, 1.0, 0, W_ + 8, ws_need, None) == S["DETFOLD_ERR_WORKSPACE"]
        assert call(arenas, 2, 64, 1.0, 0, A + 64, ws_need, None) == S["DETFOLD_ERR_OVERLAP"]
        assert call(_tab(A, A), 2, 64, 1.0, 0, W_, ws_need, None) == S["DETFOLD_ERR_OVERLAP"]
        assert call(None, 2, 64, 1.0, 0, W_, ws_need, None) == S["DETFOLD_ERR_NULL"]
        assert call(arenas, 0, 64, 1.0, 0, W_, ws_need, None) == S["DETFOLD_ERR_WORLD"]
        assert call(arenas, 2, 0, 0.5, 0, None, 0, None) == S["DETFOLD_OK"]


@no_gpu_only
def test_validation_broadcast_and_all_gather(df):
    L, S = df.lib, df.STATUS
    assert L.detfold_broadcast(None, 2, A, 8, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_broadcast(_tab(A, A + 4096), 2, None, 8, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_broadcast(_tab(A, A + 4096), 0, A + 8192, 8, None) == S["DETFOLD_ERR_WORLD"]
    assert L.detfold_broadcast(_tab(A, A + 4096), 2, A + 8194, 8, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_broadcast(_tab(A, A + 16), 2, A + 8192, 8, None) == S["DETFOLD_ERR_OVERLAP"]
    assert L.detfold_broadcast(_tab(A, A + 4096), 2, A + 4, 8, None) == S["DETFOLD_ERR_OVERLAP"]
    assert L.detfold_broadcast(_tab(A, A + 4096), 2, A + 8192, 0, None) == S["DETFOLD_OK"]
    outs = _tab(A, A + 4096)
    parts = _tab(A + 8192, A + 8192 + 64)
    assert L.detfold_all_gather(None, 2, parts, 8, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_all_gather(outs, 0, parts, 8, None) == S["DETFOLD_ERR_WORLD"]
    assert L.detfold_all_gather(outs, 2, parts, -1, None) == S["DETFOLD_ERR_LEN"]
    assert L.detfold_all_gather(_tab(A, A + 32), 2, parts, 8, None) == S["DETFOLD_ERR_OVERLAP"]
    assert L.detfold_all_gather(outs, 2, _tab(A + 8, A + 8192), 8, None) == S["DETFOLD_ERR_OVERLAP"]
    assert L.detfold_all_gather(outs, 2, _tab(A + 8194, A + 8192), 8, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_all_gather(outs, 2, parts, 0, None) == S["DETFOLD_OK"]


@no_gpu_only
def test_validation_device_tables(df):
    L, S = df.lib, df.STATUS
    T = A + (1 << 16)  # a fake 8-byte-aligned device table address
    assert L.detfold_sum_ptrs_dev(None, T, 2, 8, None, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_sum_ptrs_dev(A, None, 2, 8, None, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_sum_ptrs_dev(A, T, 0, 8, None, None) == S["DETFOLD_ERR_WORLD"]
    assert L.detfold_sum_ptrs_dev(A, T, 2, -2, None, None) == S["DETFOLD_ERR_LEN"]
    assert L.detfold_sum_ptrs_dev(A, T + 4, 2, 8, None, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_sum_ptrs_dev(A + 2, T, 2, 8, None, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_sum_ptrs_dev(A, T, 2, 8, A + 6, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_sum_ptrs_dev(A, T, 2, 0, None, None) == S["DETFOLD_OK"]
    assert L.detfold_loopback_allreduce_dev(None, 2, 8, 1.0, None, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_loopback_allreduce_dev(T, 300, 8, 1.0, None, None) == S["DETFOLD_ERR_WORLD"]
    assert L.detfold_loopback_allreduce_dev(T + 2, 2, 8, 1.0, None, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_loopback_allreduce_dev(T, 1, 8, 1.0, None, None) == S["DETFOLD_OK"]
    assert L.detfold_loopback_allreduce_dev(T, 2, 0, 0.5, None, None) == S["DETFOLD_OK"]


@no_gpu_only
def test_validation_one_shot(df):
    L, S = df.lib, df.STATUS
    arenas = _tab(A, A + 4096)
    link, stage, words = A + (1 << 20), A + (1 << 21), A + (1 << 22)
    ok = dict(link=link, epoch=1, stage=stage, words=words, wait=1000000, drop=-1, at_exit=0)

    def call(arenas=arenas, W=2, n=64, **kw):
        a = {**ok, **kw}
        return L.detfold_one_shot_allreduce(arenas, W, n, 1.0, a["link"], a["epoch"], a["stage"],
                                            a["words"], a["wait"], a["drop"], a["at_exit"], None)
    assert call(link=None) == S["DETFOLD_ERR_NULL"]
    assert call(stage=None) == S["DETFOLD_ERR_NULL"]
    assert call(words=None) == S["DETFOLD_ERR_NULL"]
    assert call(W=0) == S["DETFOLD_ERR_WORLD"]
    assert call(W=65) == S["DETFOLD_ERR_WORLD"]
    assert call(n=(1 << 22) + 1) == S["DETFOLD_ERR_LEN"]
    assert call(epoch=0, n=0) == S["DETFOLD_OK"]  # 0: the link's counter supplies the epoch
    # the counter sits past the barrier flags and belongs to the link
    assert call(link=A - df.DETFOLD_ONESHOT_LINK_BYTES + 32) == S["DETFOLD_ERR_OVERLAP"]
    assert call(wait=0) == S["DETFOLD_ERR_ARG"]
    assert call(wait=3_000_000_000) == S["DETFOLD_ERR_ARG"]
    assert call(drop=2) == S["DETFOLD_ERR_ARG"]
    assert call(link=link + 4) == S["DETFOLD_ERR_ALIGN"]
    assert call(arenas=_tab(A, A + 8)) == S["DETFOLD_ERR_OVERLAP"]
    assert call(stage=A + 100) == S["DETFOLD_ERR_OVERLAP"]
    assert call(n=0) == S["DETFOLD_OK"]


@no_gpu_only
def test_validation_scale(df):
    L, S = df.lib, df.STATUS
    assert L.detfold_scale(None, 8, 0.5, None) == S["DETFOLD_ERR_NULL"]
    assert L.detfold_scale(A + 1, 8, 0.5, None) == S["DETFOLD_ERR_ALIGN"]
    assert L.detfold_scale(A, -8, 0.5, None) == S["DETFOLD_ERR_LEN"]
    assert L.detfold_scale(A, 8, 1.0, None) == S["DETFOLD_OK"]   # scale 1: nothing enqueued


@no_gpu_only
def test_validation_probes(df):
    import bench
    P, S = bench.Probes().lib, df.STATUS
    assert P.detfold_probe_launch_floor(-1, 1, None) == S["DETFOLD_ERR_ARG"]
    assert P.detfold_probe_launch_floor(0, 1, None) == S["DETFOLD_OK"]
    assert P.detfold_probe_memory_floor(None, A, 1, 1, None) == S["DETFOLD_ERR_NULL"]
    assert P.detfold_probe_memory_floor(A, None, 1, 1, None) == S["DETFOLD_ERR_NULL"]
    assert P.detfold_probe_memory_floor(A, A + 128, -1, 1, None) == S["DETFOLD_ERR_ARG"]
    assert P.detfold_probe_memory_floor(A + 2, A + 128, 1, 1, None) == S["DETFOLD_ERR_ALIGN"]
    assert P.detfold_probe_memory_floor(A, A + 124, 1, 1, None) == S["DETFOLD_ERR_OVERLAP"]
    assert P.detfold_probe_memory_floor(A, A + 128, 0, 1, None) == S["DETFOLD_OK"]
    F = P.detfold_probe_same_shape_floor
    B, C = A + (1 << 20), A + (2 << 20)
    assert F(None, B, C, 4096, 1, None) == S["DETFOLD_ERR_NULL"]
    assert F(A, B, C, 4096, -1, None) == S["DETFOLD_ERR_ARG"]
    for n in (0, 1000, 4097, 4096 + 512, (1 << 17) + 1024):
        assert F(A, B, C, n, 1, None) == S["DETFOLD_ERR_LEN"], n
    assert F(A + 16, B, C, 4096, 1, None) == S["DETFOLD_ERR_ALIGN"]
    assert F(A, B + 4, C, 4096, 1, None) == S["DETFOLD_ERR_ALIGN"]
    assert F(A, A + 4096, C, 4096, 1, None) == S["DETFOLD_ERR_OVERLAP"]
    assert F(A, B, C, 4096, 0, None) == S["DETFOLD_OK"]


@no_gpu_only
def test_launch_without_device_reports_cuda_error(df):
    L, S = df.lib, df.STATUS
    rc = L.detfold_sum_stacked(A, A + 4096, 2, 8, None)
    assert rc == S["DETFOLD_ERR_CUDA"]
    assert L.detfold_last_cuda_error() != 0
    with pytest.raises(df.DetfoldError):
        df.detfold_sum_stacked(A, A + 4096, 2, 8, stream=0)


def test_binding_checks_tensor_sizes(df):
    torch = pytest.importorskip("torch")
    t = torch.zeros(8)
    with pytest.raises(TypeError):
        df.detfold_sum_stacked(t, t, 2, 4, stream=0)   # CPU tensors are refused


def test_oracle_and_library_share_no_code():
    # Neither side includes, imports or links the other.
    pkg = os.path.join(ROOT, "deterministic_fixed_order_gb300")
    banned = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#include\s+.*oracle)", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                assert not banned.search(open(os.path.join(dirpath, f)).read()), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "deterministic_fixed_order_gb300" not in text and "detfold.h" not in text, f
