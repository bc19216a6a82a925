"""One-shot all-reduce emulation (single cooperative launch, bounded barriers).

memra-engine 0.128.0 tests/tp_ar_gpu.rs, `one_shot_all_reduce_matches_the_host_sum_bitwise`:
three rounds on one link, the barrier words read first, round r giving
want * 2^r at W = 2. Failure detection without a fault: a dropped rank makes
the others' bounded waits run out, they return the refusal word and leave
their arenas untouched, and the next call on the same link works again.
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


@pytest.mark.parametrize("n", [1, 1024, 4096, 16384, 65536])
def test_three_rounds_double_the_sum(n):
    a, b = gen.vecf(n, 11 + n), gen.vecf(n, 77 + n)
    want = oracle.fold(np.stack([a, b]))
    link = df.OneShotLink(2, n)
    xa, xb = Guarded(n, 0, a), Guarded(n, 0, b)
    for rnd in range(3):
        link.all_reduce([xa.t, xb.t])
        torch.cuda.synchronize()
        # the barrier words first: an expired barrier leaves x untouched
        assert link.barrier_errors() == [0, 0], f"n={n} round={rnd}"
        w = (want.astype(np.float64) * (1 << rnd)).astype(np.float32)
        assert_bitwise(xa.host(), w, f"rank 0 n={n} round={rnd}")
        assert_bitwise(xb.host(), w, f"rank 1 n={n} round={rnd}")
        assert xa.intact() and xb.intact()


@pytest.mark.parametrize("W", [3, 4, 8, 16])
@pytest.mark.parametrize("n", [7, 4099, 100_003])
def test_matches_oracle_over_rounds(W, n):
    rows = gen.stress_rows(W, n)
    scale = float(oracle.mean_scale(W))
    arenas = [Guarded(n, r % 3, rows[r]) for r in range(W)]
    host = [rows[r].copy() for r in range(W)]
    link = df.OneShotLink(W, n)
    for rnd in range(3):
        link.all_reduce([x.t for x in arenas], scale)
        oracle.allreduce(host, np.float32(scale))
        torch.cuda.synchronize()
        assert link.barrier_errors() == [0] * W
        for r in range(W):
            assert_bitwise(arenas[r].host(), host[r], f"W={W} n={n} round={rnd} rank={r}")


@pytest.mark.parametrize("at_exit", [False, True])
def test_dropped_rank_refuses_and_leaves_arenas_untouched(at_exit):
    W, n = 4, 4096
    rows = gen.normal_rows(W, n)
    arenas = [Guarded(n, 0, rows[r]) for r in range(W)]
    link = df.OneShotLink(W, n)
    link.all_reduce([x.t for x in arenas], drop_rank=2, drop_at_exit=at_exit, wait_ns=20_000_000)
    torch.cuda.synchronize()
    words = link.barrier_errors()
    code = df.DETFOLD_ONESHOT_REFUSE_EXIT if at_exit else df.DETFOLD_ONESHOT_REFUSE_ENTRY
    assert words == [code, code, 0, code], words   # the dropped rank wrote nothing
    for r in range(W):
        assert_bitwise(arenas[r].host(), rows[r], f"rank {r} changed after a refusal")
    # the same link works again on the next epoch
    link.all_reduce([x.t for x in arenas])
    torch.cuda.synchronize()
    assert link.barrier_errors() == [0] * W
    want = [rows[r].copy() for r in range(W)]
    oracle.allreduce(want)
    for r in range(W):
        assert_bitwise(arenas[r].host(), want[r], f"rank {r} after recovery")


def test_graph_replays_take_fresh_epochs_from_the_link():
    # With the link's counter supplying the epoch, one captured call replays
    # as a fresh call each time: the three rounds double the sum, as eagerly.
    n = 4096
    a, b = gen.vecf(n, 11 + n), gen.vecf(n, 77 + n)
    want = oracle.fold(np.stack([a, b]))
    link = df.OneShotLink(2, n)
    xa, xb = Guarded(n, 0, a), Guarded(n, 0, b)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        link.all_reduce([xa.t, xb.t])
    assert link.counter() == 0  # nothing ran during the capture
    for rnd in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert link.barrier_errors() == [0, 0], f"replay {rnd}"
        assert link.counter() == rnd + 1
        w = (want.astype(np.float64) * (1 << rnd)).astype(np.float32)
        assert_bitwise(xa.host(), w, f"rank 0 replay {rnd}")
        assert_bitwise(xb.host(), w, f"rank 1 replay {rnd}")
    # a graph of several calls: each node takes the next epoch
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        for _ in range(4):
            link.all_reduce([xa.t, xb.t])
    g2.replay()
    torch.cuda.synchronize()
    assert link.counter() == 3 + 4
    w = (want.astype(np.float64) * (1 << 6)).astype(np.float32)
    assert_bitwise(xa.host(), w, "after a 4-call graph")
    assert xa.intact() and xb.intact()


def test_host_and_device_epochs_mix_on_one_link():
    W, n = 3, 1000
    rows = gen.normal_rows(W, n)
    arenas = [Guarded(n, 0, rows[r]) for r in range(W)]
    host = [rows[r].copy() for r in range(W)]
    link = df.OneShotLink(W, n)
    link.all_reduce([x.t for x in arenas])           # device epoch 1
    link.all_reduce([x.t for x in arenas], epoch=5)  # host epoch above the counter
    torch.cuda.synchronize()
    assert link.counter() == 5  # raised to the host's epoch
    link.all_reduce([x.t for x in arenas])           # device epoch 6
    torch.cuda.synchronize()
    assert link.counter() == 6
    assert link.barrier_errors() == [0] * W
    for _ in range(3):
        oracle.allreduce(host)
    for r in range(W):
        assert_bitwise(arenas[r].host(), host[r], f"rank {r}")


def test_refused_call_advances_the_counter():
    # Every CTA raises the counter to the epoch it used, so the next call's
    # epoch is above every flag a refused call left behind. A rank dropped at
    # the entry leaves at once; a CTA that reads the counter after that takes
    # the next epoch, so the counter may advance by two. A rank dropped at the
    # exit leaves only after every CTA has read the counter: exactly one.
    W, n = 4, 4096
    rows = gen.normal_rows(W, n)
    arenas = [Guarded(n, 0, rows[r]) for r in range(W)]
    link = df.OneShotLink(W, n)
    for at_exit in (False, True):
        before = link.counter()
        link.all_reduce([x.t for x in arenas], drop_rank=1, drop_at_exit=at_exit, wait_ns=20_000_000)
        torch.cuda.synchronize()
        if at_exit:
            assert link.counter() == before + 1
        else:
            assert before + 1 <= link.counter() <= before + 2
        for r in range(W):
            assert_bitwise(arenas[r].host(), rows[r], f"rank {r} changed after a refusal")
    link.all_reduce([x.t for x in arenas])
    torch.cuda.synchronize()
    assert link.barrier_errors() == [0] * W
    want = [rows[r].copy() for r in range(W)]
    oracle.allreduce(want)
    for r in range(W):
        assert_bitwise(arenas[r].host(), want[r], f"rank {r} after the refusals")
