"""The bulk-async (TMA) staged bandwidth path, at and around its thresholds.

Large aligned folds and all-reduces (W <= 8, len >= 2^20, every operand at
one 16-byte phase) stream tiles through shared memory with cp.async.bulk.
The per-element chain is the same (mamba-rs 0.6.2 src/dist/reducer.rs,
`reduce_sum_reference`), so the bits must equal the oracle's; the head
before the first tile and the ragged tail after the last take scalar code in
the same launch. Every bounded pipeline wait must have succeeded.
"""
import numpy as np
import pytest
import torch

import detfold_inputs as gen
import oracle
from gpu_util import Guarded, assert_bitwise

import deterministic_fixed_order_gb300 as df

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

M = 1 << 21  # the fold's bulk-async threshold (DETFOLD_BULK_MIN_LEN)


@pytest.mark.parametrize("W", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n", [M, M + 1, M + 4099, 3 * M + 12345])
def test_bulk_allreduce_arenas_at_different_16_byte_phases(W, n):
    # The all-reduce whose arenas do not share a 16-byte phase takes the
    # bulk-async pipeline with per-arena offsets at these sizes: each arena
    # must end with the oracle's bits, guard bands intact, no wait expired.
    rng = np.random.default_rng(31 * W + n % 1009)
    offs = [int(x) for x in rng.integers(0, 8, size=W)]
    if len({o % 4 for o in offs}) == 1:
        offs[-1] = (offs[-1] + 1) % 8  # at least two 16-byte phases
    rows = gen.stress_rows(W, n, seed0=int(rng.integers(1, 1 << 30)))
    scale = float(oracle.mean_scale(W))
    arenas = [Guarded(n, offs[r], rows[r]) for r in range(W)]
    df.detfold_loopback_allreduce([a.t for a in arenas], W, n, scale)
    torch.cuda.synchronize()
    want = [rows[r].copy() for r in range(W)]
    oracle.allreduce(want, np.float32(scale))
    for r in range(W):
        assert arenas[r].intact(), f"guard band of arena {r} (offsets {offs})"
        assert_bitwise(arenas[r].host(), want[r], f"mixed-phase bulk all-reduce W={W} n={n} offs={offs} rank {r}")
    assert df.detfold_pipeline_timeouts() == 0


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n", [M, M + 1, M + 2047, M + 4099, 3 * M + 12345])
def test_bulk_sum_and_allreduce(W, n):
    rows = gen.stress_rows(W, n)
    want = oracle.fold(rows)
    # sum into a separate output, all operands 32-byte aligned
    srcs = [Guarded(n, 0, rows[r]) for r in range(W)]
    out = Guarded(n)
    df.detfold_sum_ptrs(out.t, [s.t for s in srcs], W, n)
    torch.cuda.synchronize()
    assert_bitwise(out.host(), want, f"bulk sum W={W} n={n}")
    assert out.intact()
    # all operands at the same odd phase: a scalar head, then 32-byte tiles
    srcs3 = [Guarded(n, 3, rows[r]) for r in range(W)]
    out3 = Guarded(n, 3)
    df.detfold_sum_ptrs(out3.t, [s.t for s in srcs3], W, n)
    torch.cuda.synchronize()
    assert_bitwise(out3.host(), want, f"bulk sum phase 3 W={W} n={n}")
    # a shared 16-byte (not 32-byte) phase: offsets 0 and 4 elements mixed
    srcs4 = [Guarded(n, 4 * (r % 2), rows[r]) for r in range(W)]
    out4 = Guarded(n, 4)
    df.detfold_sum_ptrs(out4.t, [s.t for s in srcs4], W, n)
    torch.cuda.synchronize()
    assert_bitwise(out4.host(), want, f"bulk sum 16-byte phase W={W} n={n}")
    # in place: out is the last source
    df.detfold_sum_ptrs(srcs[-1].t, [s.t for s in srcs], W, n)
    torch.cuda.synchronize()
    assert_bitwise(srcs[-1].host(), want, f"bulk in-place W={W} n={n}")
    # fused all-reduce with the mean
    scale = float(oracle.mean_scale(W))
    arenas = [Guarded(n, 1, rows[r]) for r in range(W)]
    df.detfold_loopback_allreduce([a.t for a in arenas], W, n, scale)
    torch.cuda.synchronize()
    mean = oracle.scale(want, scale)
    for r in range(W):
        assert_bitwise(arenas[r].host(), mean, f"bulk all-reduce W={W} n={n} rank={r}")
        assert arenas[r].intact()


@pytest.mark.parametrize("n", [M, M + 4099, 3 * M + 12345])
@pytest.mark.parametrize("off", [0, 1, 2, 3])
def test_bulk_scale_pass_matches_the_oracle(n, off):
    # The separate mean pass at bulk sizes (a W=1 all-reduce on the bulk
    # pipeline, with its own deeper tile shape): fl(x * s) element by element,
    # at every 16-byte phase of the buffer, guard bands intact.
    row = gen.stress_rows(1, n, seed0=5 + off)[0]
    s = float(oracle.mean_scale(3))
    buf = Guarded(n, off, row)
    df.detfold_scale(buf.t, n, s)
    torch.cuda.synchronize()
    assert buf.intact()
    assert_bitwise(buf.host(), oracle.scale(row, s), f"scale n={n} off={off}")
    assert df.detfold_pipeline_timeouts() == 0


def test_bulk_repeated_calls_and_no_pipeline_timeouts():
    W, n = 4, 5 * M + 777
    rows = gen.normal_rows(W, n)
    arenas = [Guarded(n, 0, rows[r]) for r in range(W)]
    host = [rows[r].copy() for r in range(W)]
    for _ in range(5):
        df.detfold_loopback_allreduce([a.t for a in arenas], W, n, 0.25)
        oracle.allreduce(host, np.float32(0.25))
    torch.cuda.synchronize()
    for r in range(W):
        assert_bitwise(arenas[r].host(), host[r], f"repeated bulk all-reduce rank {r}")
    assert df.detfold_pipeline_timeouts() == 0


def _bits_rows(W, n, seed):
    return np.random.default_rng(seed).integers(0, 2 ** 32, size=(W, n), dtype=np.uint64) \
        .astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("n", [M, M + 5, M + 2047, M + 2053, 3 * M + 2049])
@pytest.mark.parametrize("nd", [1, 3, 7])
def test_bulk_broadcast_moves_bytes_exactly(n, nd):
    # offset 2: a 2-element head; M + 2047 and M + 2053 leave tails of 2045
    # and 3 elements after the 8 KB tiles (16-byte vectors, then scalars)
    src_h = _bits_rows(1, n, n + nd)[0]
    src = Guarded(n, 2, src_h)
    dsts = [Guarded(n, 2) for _ in range(nd)]
    df.detfold_broadcast([d.t for d in dsts], nd, src.t, n)
    torch.cuda.synchronize()
    for k, d in enumerate(dsts):
        assert_bitwise(d.host(), src_h, f"bulk broadcast n={n} dst={k}")
        assert d.intact()


@pytest.mark.parametrize("W", [2, 4, 5, 8])
def test_bulk_all_gather_and_staged(W):
    span = M + 4  # keeps every part's offset at the same 16-byte phase
    parts_h = _bits_rows(W, span, 100 + W)
    parts = [Guarded(span, 0, parts_h[r]) for r in range(W)]
    outs = [Guarded(W * span, 0) for _ in range(W)]
    df.detfold_all_gather([o.t for o in outs], W, [p.t for p in parts], span)
    torch.cuda.synchronize()
    want = parts_h.reshape(-1)
    for r, o in enumerate(outs):
        assert_bitwise(o.host(), want, f"bulk all-gather W={W} rank={r}")
        assert o.intact()
    # the staged comparator with shards of at least 2^20: bulk exchange and
    # distribute, with shard tails of about 2000 elements after the tiles
    n = W * (M + 2000) + 13
    rows = gen.normal_rows(W, n)
    arenas = [Guarded(n, 1, rows[r]) for r in range(W)]
    nb = df.detfold_staged_workspace_bytes(n, W)
    ws = torch.empty(nb // 4, dtype=torch.float32, device="cuda")
    scale = float(oracle.mean_scale(W))
    for flags in (0, 1, 2):
        for r in range(W):
            arenas[r].t.copy_(torch.from_numpy(rows[r]))
        df.detfold_loopback_allreduce_staged_ex([a.t for a in arenas], W, n, scale, flags, ws, nb)
        torch.cuda.synchronize()
        want = [rows[r].copy() for r in range(W)]
        oracle.allreduce(want, np.float32(scale))
        for r in range(W):
            assert_bitwise(arenas[r].host(), want[r], f"bulk staged W={W} flags={flags} rank={r}")
            assert arenas[r].intact()
    assert df.detfold_pipeline_timeouts() == 0


def test_first_use_inside_graph_capture(tmp_path):
    # A fresh process whose first bulk/movement/realign launches are captured.
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = str(tmp_path / "res.npy")
    r = subprocess.run([sys.executable, os.path.join(root, "tests", "helpers", "capture_first_use.py"),
                        root, out], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "timeouts 0" in r.stdout
    res = np.load(out)
    W, n = 4, (1 << 22) + 5
    rows = gen.stress_rows(W, n)
    assert_bitwise(res[0], oracle.fold(rows), "captured ptrs fold")
    want = [rows[q].copy() for q in range(W)]
    oracle.allreduce(want, np.float32(0.25))
    for k, q in ((1, 0), (2, W - 1), (3, 0), (4, W - 1), (5, 0), (6, W - 1)):
        assert_bitwise(res[k], want[q], f"captured all-reduce result {k}")
