"""libdetfold used from plain C through include/detfold.h, with no Python in
the loop: a host-only program on the CPU, and a device program on the GPU
whose outputs are checked against the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import detfold_inputs as gen
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.join(ROOT, "tests", "c_consumer")
INC = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "deterministic_fixed_order_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(src, out, cflags=(), ldflags=()):
    # libraries after the source: some linkers resolve them in order
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Werror", "-I", INC, *cflags,
           os.path.join(HERE, src), "-o", out, "-L", PKG, "-ldetfold", f"-Wl,-rpath,{PKG}",
           *ldflags]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_host_only_c_program(tmp_path):
    exe = str(tmp_path / "host_only")
    _build("host_only.c", exe)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    lines = dict(l.split(" ", 1) for l in r.stdout.splitlines() if not l.startswith("shard"))
    shards = [l.split()[1:] for l in r.stdout.splitlines() if l.startswith("shard")]
    starts, lens = oracle.shard_plan((1 << 20) + 7, 6)
    assert [[int(a), int(b), int(c)] for a, b, c in shards] == \
        [[r, int(s), int(n)] for r, (s, n) in enumerate(zip(starts, lens))]
    assert int(lines["ws"]) >= 4 * (25_000_000 + 8) * 4
    assert int(lines["null"]) == -1 and int(lines["world"]) == -2 and int(lines["zero"]) == 0
    assert "overlap" in lines["str"]


@pytest.mark.gpu
def test_device_c_program_matches_oracle(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("CUDA headers not found")
    exe = str(tmp_path / "device_fold")
    _build("device_fold.c", exe, cflags=["-I", os.path.join(CUDA, "include")],
           ldflags=["-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"])
    # realigned and bulk-async paths, the small path, the 16 KiB decode join
    # (exact small grid) and an aligned stack on the bulk path
    for W, n in ((3, (1 << 20) + 7), (4, 100_003), (8, 4099), (2, 4096), (4, (1 << 20) + 4096)):
        rows = gen.stress_rows(W, n)
        inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
        rows.tofile(inp)
        scale = float(oracle.mean_scale(W))
        r = subprocess.run([exe, str(inp), str(outp), str(W), repr(scale)], capture_output=True,
                           text=True, timeout=120)
        assert r.returncode == 0, r.stderr
        got = np.fromfile(outp, dtype=np.float32).reshape(W + 1, n)
        want = oracle.fold(rows)
        assert oracle.bit_diffs(got[0], want) == 0, f"C fold W={W}"
        arenas = [rows[q].copy() for q in range(W)]
        oracle.allreduce(arenas, np.float32(scale))
        for q in range(W):
            assert oracle.bit_diffs(got[1 + q], arenas[q]) == 0, f"C all-reduce W={W} rank {q}"
