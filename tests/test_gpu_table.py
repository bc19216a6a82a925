"""Device-resident pointer tables and CUDA-graph rebind.

The rebind gate of memra-engine 0.136.0 tests/gdn_packed_gpu.rs captures a
graph once, rewrites the device pointer table, replays, and requires the
bits of a fresh eager run -- including after swapping the canonical and
alternate addresses. Here the table feeds the fixed-order fold (mamba-rs
0.6.2 src/dist/reducer.rs, `reduce_sum_reference`), checked against the oracle.
"""
import numpy as np
import pytest
import torch

import detfold_inputs as gen
import oracle
from gpu_util import SENTINEL, Guarded, assert_bitwise

import deterministic_fixed_order_gb300 as df

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def sync():
    torch.cuda.synchronize()


@pytest.mark.parametrize("W", [1, 2, 3, 4, 8, 9, 33])
@pytest.mark.parametrize("n", [1, 4096, 4099, (1 << 20) + 7])
@pytest.mark.parametrize("phases", ["aligned", "mixed"])
def test_table_fold_matches_oracle(W, n, phases):
    rows = gen.stress_rows(W, n)
    offs = [0] * W if phases == "aligned" else [(3 * r) % 8 for r in range(W)]
    srcs = [Guarded(n, offs[r], rows[r]) for r in range(W)]
    out = Guarded(n, 0 if phases == "aligned" else 5)
    table = df.device_table([s.t for s in srcs])
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    df.detfold_sum_ptrs_dev(out.t, table, W, n, status)
    sync()
    assert int(status.item()) == 0
    assert_bitwise(out.host(), oracle.fold(rows), f"table fold W={W} n={n} {phases}")
    assert out.intact() and all(s.intact() for s in srcs)


# per-rank element offsets -> the access width the kernel must pick
PHASE_PLANS = {
    "32B+head": lambda r: 5,            # one 32-byte phase, head 3
    "16B": lambda r: 4 * (r % 2),       # 16-byte phase shared, 32-byte phase not
    "16B+head": lambda r: 1 + 4 * (r % 2),
    "scalar": lambda r: r % 4,
}


@pytest.mark.parametrize("W", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [1, 9, 1034, 4099, 65536 + 3, 1 << 17, (1 << 17) + 1,
                               (1 << 20) + 7, (1 << 21) + 2047])
@pytest.mark.parametrize("plan", sorted(PHASE_PLANS))
def test_table_access_widths_heads_and_tails(W, n, plan):
    # The table kernels choose the access width on the device from the
    # entries' phases; every width, with heads and tails, on both sides of
    # the small-payload bound (2^17 elements) and past the bulk bound (2^20,
    # where one 16-byte phase runs the bulk pipeline fed from the table and
    # mixed phases a scalar fold), for the sum, the in-place sum and the
    # all-reduce.
    rows = gen.stress_rows(W, n)
    offs = [PHASE_PLANS[plan](r) for r in range(W)]
    srcs = [Guarded(n, offs[r], rows[r]) for r in range(W)]
    out = Guarded(n, offs[0])
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    df.detfold_sum_ptrs_dev(out.t, df.device_table([t.t for t in srcs]), W, n, status)
    sync()
    assert int(status.item()) == 0
    want = oracle.fold(rows)
    assert_bitwise(out.host(), want, f"table fold W={W} n={n} {plan}")
    assert out.intact() and all(t.intact() for t in srcs)
    df.detfold_sum_ptrs_dev(srcs[0].t, df.device_table([t.t for t in srcs]), W, n)
    sync()
    assert_bitwise(srcs[0].host(), want, f"table in-place W={W} n={n} {plan}")
    scale = float(oracle.mean_scale(W))
    arenas = [Guarded(n, offs[r], rows[r]) for r in range(W)]
    df.detfold_loopback_allreduce_dev(df.device_table([a.t for a in arenas]), W, n, scale)
    sync()
    exp = [rows[r].copy() for r in range(W)]
    oracle.allreduce(exp, np.float32(scale))
    for r in range(W):
        assert_bitwise(arenas[r].host(), exp[r], f"table all-reduce W={W} n={n} {plan} rank={r}")
        assert arenas[r].intact()


@pytest.mark.parametrize("W", [2, 3, 4, 6])
@pytest.mark.parametrize("n", [5, 65536 + 3, (1 << 20) + 7])
def test_table_allreduce_and_in_place_fold(W, n):
    rows = gen.normal_rows(W, n)
    scale = float(oracle.mean_scale(W))
    arenas = [Guarded(n, r % 4, rows[r]) for r in range(W)]
    df.detfold_loopback_allreduce_dev(df.device_table([a.t for a in arenas]), W, n, scale)
    sync()
    want = [rows[r].copy() for r in range(W)]
    oracle.allreduce(want, np.float32(scale))
    for r in range(W):
        assert_bitwise(arenas[r].host(), want[r], f"table all-reduce W={W} rank={r}")
        assert arenas[r].intact()
    # in place: out is the last source
    srcs = [Guarded(n, 0, rows[r]) for r in range(W)]
    df.detfold_sum_ptrs_dev(srcs[-1].t, df.device_table([s.t for s in srcs]), W, n)
    sync()
    assert_bitwise(srcs[-1].host(), oracle.fold(rows), f"table in-place W={W}")


def test_graph_replay_follows_a_rebound_table():
    n, W = 4096, 3
    sets = [gen.stress_rows(W, n), gen.normal_rows(W, n)]
    bufs = [[Guarded(n, 0, rows[r]) for r in range(W)] for rows in sets]
    out = Guarded(n)
    table = df.device_table([b.t for b in bufs[0]])
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        df.detfold_sum_ptrs_dev(out.t, table, W, n)  # first call outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(20):
            df.detfold_sum_ptrs_dev(out.t, table, W, n)
    # replay 0: the capture-time table; replay 1: a new buffer set;
    # replay 2: the new set in reversed rank order (the canonical/alternate swap)
    plans = [(bufs[0], sets[0]), (bufs[1], sets[1]),
             (bufs[1][::-1], np.ascontiguousarray(sets[1][::-1]))]
    results = []
    for bset, rows in plans:
        table.copy_(df.device_table([b.t for b in bset]))
        out.t.zero_()
        g.replay()
        sync()
        got = out.host()
        assert_bitwise(got, oracle.fold(rows), "graph replay after rebind")
        assert out.intact()
        results.append(got)
    # the reversed order is a different fold: some bits differ (stress data)
    assert oracle.bit_diffs(results[1], results[2]) > 0


def test_table_status_reports_bad_entries_and_writes_nothing():
    n, W = 1000, 3
    rows = gen.normal_rows(W, n)
    srcs = [Guarded(n, 0, rows[r]) for r in range(W)]
    out = Guarded(n)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptrs = [s.t.data_ptr() for s in srcs]
    cases = {
        "null": ([ptrs[0], 0, ptrs[2]], df.STATUS["DETFOLD_ERR_NULL"]),
        "misaligned": ([ptrs[0], ptrs[1] + 2, ptrs[2]], df.STATUS["DETFOLD_ERR_ALIGN"]),
    }
    for name, (entries, code) in cases.items():
        table = torch.tensor(entries, dtype=torch.int64, device="cuda")
        df.detfold_sum_ptrs_dev(out.t, table, W, n, status)   # host returns OK: launch ran
        df.detfold_loopback_allreduce_dev(table, W, n, 0.5, status)
        sync()
        assert int(status.item()) == code, name
        # nothing written: out still holds the sentinel, sources unchanged
        assert bool((out.t.view(torch.int32) == SENTINEL).all()), name
        for r in range(W):
            assert_bitwise(srcs[r].host(), rows[r], f"{name}: source {r} changed")
    table = df.device_table([s.t for s in srcs])
    df.detfold_sum_ptrs_dev(out.t, table, W, n, status)
    sync()
    assert int(status.item()) == 0
    assert_bitwise(out.host(), oracle.fold(rows), "valid table after bad ones")
