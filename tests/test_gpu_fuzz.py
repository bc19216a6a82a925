"""Seeded random parity cases across the dispatch boundaries.

Each case draws a world size, a length, per-operand 4-byte phases and an entry
point, runs it through the library and compares every written word with the
oracle (0 ULP), with guard bands checked. Lengths cluster at the boundaries
where the dispatch changes kernels: the small-payload bound (2^17 elements),
the bulk-async bound (2^20), whole tiles (2048 and 1024 floats per rank) and
the vector widths (4 and 8 floats). The case list is fixed by the seed, so a
failure names a reproducible case.
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

# the small-payload bound; the bulk-async bounds of table folds and moves
# (2^20) and of parameter-table folds (2^21)
SMALL, BULK, BULK2 = 1 << 17, 1 << 20, 1 << 21
BOUNDARIES = [1, 3, 4, 7, 8, 9, 1023, 1024, 1025, 2047, 2048, 2049, 4096 + 5,
              SMALL - 1, SMALL, SMALL + 1, SMALL + 7,
              BULK - 1, BULK, BULK + 1, BULK + 7, BULK + 1023, BULK + 2047, BULK + 2048, BULK + 4095,
              BULK2 - 1, BULK2, BULK2 + 7, BULK2 + 2047, BULK2 + 4095]
ENTRIES = ["stacked", "ptrs", "in_place", "allreduce", "staged", "table_sum", "table_allreduce",
           "broadcast", "all_gather", "one_shot", "staged_noalloc"]


def _cases(count=480, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for k in range(count):
        entry = ENTRIES[k % len(ENTRIES)]
        W = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 12]))
        n = int(rng.choice(BOUNDARIES)) if rng.random() < 0.7 else int(np.exp(rng.uniform(0, np.log(3 * BULK))))
        if entry == "all_gather":
            n = min(n, BULK + 4095)
        if entry == "staged_noalloc":  # within the library's 16 MiB of scratch
            n = min(n, 600_000)
        phase = rng.random()
        if phase < 0.4:      # every operand at one phase
            off = int(rng.integers(0, 8))
            offs = [off] * (W + 1)
        elif phase < 0.6:    # one 16-byte phase, mixed 32-byte phases
            base = int(rng.integers(0, 4))
            offs = [base + 4 * int(rng.integers(0, 2)) for _ in range(W + 1)]
        else:                # independent phases
            offs = [int(x) for x in rng.integers(0, 8, size=W + 1)]
        out.append((k, entry, W, n, offs, int(rng.integers(1, 1 << 30))))
    return out


CASES = _cases()


def _rows(W, n, seed):
    # the shared seeded generators: stress (signed zeros, subnormals, 34
    # decades), gradient-like or normal values, chosen by the case's seed
    kind = (gen.stress_rows, gen.gradient_rows, gen.normal_rows)[seed % 3]
    return kind(W, n, seed0=seed)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}-W{c[2]}-n{c[3]}")
def test_random_case_matches_oracle(case):
    k, entry, W, n, offs, seed = case
    rows = _rows(W, n, seed)
    what = f"case {k}: {entry} W={W} n={n} offsets={offs}"
    if entry == "stacked":
        st = Guarded(W * n, offs[0], rows)
        out = Guarded(n, offs[1])
        df.detfold_sum_stacked(out.t, st.t, W, n)
        torch.cuda.synchronize()
        assert st.intact() and out.intact(), what
        assert_bitwise(out.host(), oracle.fold(rows), what)
    elif entry in ("ptrs", "in_place", "table_sum"):
        srcs = [Guarded(n, offs[r], rows[r]) for r in range(W)]
        if entry == "in_place":
            out = srcs[W // 2]
        else:
            out = Guarded(n, offs[W])
        if entry == "table_sum":
            df.detfold_sum_ptrs_dev(out.t, df.device_table([s.t for s in srcs]), W, n)
        else:
            df.detfold_sum_ptrs(out.t, [s.t for s in srcs], W, n)
        torch.cuda.synchronize()
        assert out.intact() and all(s.intact() for s in srcs), what
        assert_bitwise(out.host(), oracle.fold(rows), what)
    elif entry in ("allreduce", "staged", "table_allreduce", "one_shot", "staged_noalloc"):
        scale = float(oracle.mean_scale(W)) if seed % 2 else 1.0
        arenas = [Guarded(n, offs[r], rows[r]) for r in range(W)]
        ts = [a.t for a in arenas]
        if entry == "allreduce":
            df.detfold_loopback_allreduce(ts, W, n, scale)
        elif entry == "table_allreduce":
            df.detfold_loopback_allreduce_dev(df.device_table(ts), W, n, scale)
        elif entry == "one_shot":
            link = df.OneShotLink(W, n)
            link.all_reduce(ts, scale)
            torch.cuda.synchronize()
            assert link.barrier_errors() == [0] * W, what
        elif entry == "staged_noalloc":
            df.detfold_loopback_allreduce_staged_noalloc(ts, W, n, scale, seed % 8)
        else:
            nb = df.detfold_staged_workspace_bytes(n, W)
            ws = torch.empty(max(1, nb // 4), dtype=torch.float32, device="cuda")
            df.detfold_loopback_allreduce_staged_ex(ts, W, n, scale, seed % 8, ws, nb)
        torch.cuda.synchronize()
        want = [rows[r].copy() for r in range(W)]
        oracle.allreduce(want, np.float32(scale))
        for r in range(W):
            assert arenas[r].intact(), what
            assert_bitwise(arenas[r].host(), want[r], f"{what} rank {r}")
    elif entry == "broadcast":
        src = Guarded(n, offs[0], rows[0])
        dsts = [Guarded(n, offs[1 + r]) for r in range(W)]
        df.detfold_broadcast([d.t for d in dsts], W, src.t, n)
        torch.cuda.synchronize()
        for r, d in enumerate(dsts):
            assert d.intact(), what
            assert_bitwise(d.host(), rows[0], f"{what} dst {r}")
    else:  # all_gather
        parts = [Guarded(n, offs[r], rows[r]) for r in range(W)]
        outs = [Guarded(W * n, offs[W]) for _ in range(W)]
        df.detfold_all_gather([o.t for o in outs], W, [p.t for p in parts], n)
        torch.cuda.synchronize()
        want = rows.reshape(-1)
        for r, o in enumerate(outs):
            assert o.intact(), what
            assert_bitwise(o.host(), want, f"{what} rank {r}")
    assert df.detfold_pipeline_timeouts() == 0, what
