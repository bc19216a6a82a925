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

M = 1 << 20


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
