"""Every entry point inside CUDA-graph capture, and concurrent host threads.

A call that synchronizes or allocates device memory fails stream capture, so
capturing each entry point checks the ABI's rule that calls never sync and
never allocate. The replayed graph must reproduce the eager call's bits
exactly; the eager bits are checked against the oracle elsewhere. The
threads test drives the library from several host threads at once, each on
its own stream. That exercises the launch plumbing's per-kernel caches
(atomics) and the thread-local error slot under concurrency. The results must
match the oracle.
"""
import threading

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


class Case:
    """Inputs that reset() restores, a call() that enqueues one API call on
    the current stream, and read() of every buffer the call writes."""

    def __init__(self, rows, offsets, n_out=None, out_offset=0):
        self.rows = rows
        W, n = rows.shape
        self.W, self.n = W, n
        self.ins = [Guarded(n, offsets[r], rows[r]) for r in range(W)]
        self.out = Guarded(n if n_out is None else n_out, out_offset)
        self.host = [torch.from_numpy(np.ascontiguousarray(rows[r])) for r in range(W)]

    def reset(self):
        for t, h in zip(self.ins, self.host):
            t.t.copy_(h)
        self.out.t.zero_()

    def read(self):
        assert self.out.intact() and all(t.intact() for t in self.ins)
        return [self.out.host()] + [t.host() for t in self.ins]


def _cases():
    c = {}
    c["sum_stacked_small"] = lambda: _stacked(gen.c1_rows(2, 4096))
    c["sum_stacked_bulk"] = lambda: _stacked(gen.gradient_rows(4, M + 2047))

    def ptrs(rows, offs, out_off):
        k = Case(rows, offs, out_offset=out_off)
        k.call = lambda: df.detfold_sum_ptrs(k.out.t, [t.t for t in k.ins], k.W, k.n)
        return k
    c["sum_ptrs_realign"] = lambda: ptrs(gen.stress_rows(3, 100_003), [0, 1, 2], 5)
    c["sum_ptrs_bulk_phase3"] = lambda: ptrs(gen.stress_rows(6, M + 1029), [3] * 6, 3)

    def scale():
        k = Case(gen.normal_rows(1, M + 5), [1])
        k.call = lambda: df.detfold_scale(k.ins[0].t, k.n, 1.0 / 3.0)
        return k
    c["scale"] = scale

    def allreduce(rows, offs, s):
        k = Case(rows, offs, n_out=1)
        k.call = lambda: df.detfold_loopback_allreduce([t.t for t in k.ins], k.W, k.n, s)
        return k
    c["allreduce_bulk"] = lambda: allreduce(gen.stress_rows(3, M + 7), [1] * 3,
                                            float(oracle.mean_scale(3)))
    c["allreduce_small_mixed"] = lambda: allreduce(gen.normal_rows(5, 9999), [0, 1, 2, 3, 4], 1.0)
    c["allreduce_bulk_mixed"] = lambda: allreduce(gen.stress_rows(4, M + 4099), [0, 3, 6, 1],
                                                  float(oracle.mean_scale(4)))

    def staged(flags, W, n):
        k = Case(gen.normal_rows(W, n), [1] * W, n_out=1)
        nb = df.detfold_staged_workspace_bytes(n, W)
        k.ws = torch.empty(max(1, nb // 4), dtype=torch.float32, device="cuda")
        k.call = lambda: df.detfold_loopback_allreduce_staged_ex([t.t for t in k.ins], W, n,
                                                                  float(oracle.mean_scale(W)), flags,
                                                                  k.ws, nb)
        return k
    c["staged_sm"] = lambda: staged(0, 4, 4 * M + 13)
    c["staged_ce_copies"] = lambda: staged(4, 4, 4 * M + 13)
    c["staged_reverse_separate"] = lambda: staged(3, 3, 30_011)

    def noalloc():
        k = Case(gen.normal_rows(2, 100_000), [0, 0], n_out=1)
        k.call = lambda: df.detfold_loopback_allreduce_staged_noalloc([t.t for t in k.ins], 2, k.n, 0.5)
        return k
    c["staged_noalloc"] = noalloc

    def table(all_reduce):
        k = Case(gen.stress_rows(3, 4099), [0, 4, 0])
        k.table = df.device_table([t.t for t in k.ins])
        if all_reduce:
            k.call = lambda: df.detfold_loopback_allreduce_dev(k.table, 3, k.n, 1.0)
        else:
            k.call = lambda: df.detfold_sum_ptrs_dev(k.out.t, k.table, 3, k.n)
        return k
    c["sum_ptrs_dev"] = lambda: table(False)
    c["allreduce_dev"] = lambda: table(True)

    def broadcast():
        k = Case(gen.stress_rows(4, M + 2047), [2] * 4, n_out=1)
        k.call = lambda: df.detfold_broadcast([t.t for t in k.ins[1:]], 3, k.ins[0].t, k.n)
        return k
    c["broadcast"] = broadcast

    def all_gather():
        span = 5000
        k = Case(gen.stress_rows(3, span), [0, 0, 0], n_out=3 * 3 * span)
        outs = [k.out.t[r * 3 * span:(r + 1) * 3 * span] for r in range(3)]
        k.call = lambda: df.detfold_all_gather(outs, 3, [t.t for t in k.ins], span)
        return k
    c["all_gather"] = all_gather
    return c


def _stacked(rows):
    W, n = rows.shape
    k = Case(rows.reshape(1, -1), [0], n_out=n)
    k.call = lambda: df.detfold_sum_stacked(k.out.t, k.ins[0].t, W, n)
    return k


CASES = _cases()


@pytest.mark.parametrize("name", sorted(CASES))
def test_entry_point_inside_graph_capture(name):
    k = CASES[name]()
    k.reset()
    k.call()
    torch.cuda.synchronize()
    eager = k.read()
    assert any(np.count_nonzero(a) for a in eager), "vacuous: every output is zero"
    stream = torch.cuda.Stream()
    k.reset()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):  # fails if the call syncs or allocates
        k.call()
    for _ in range(2):
        k.reset()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for r, (got, want) in enumerate(zip(k.read(), eager)):
            assert_bitwise(got, want, f"{name}: buffer {r} after replay")
    assert df.detfold_pipeline_timeouts() == 0


def test_concurrent_host_threads_on_their_own_streams():
    n_threads, iters = 4, 60
    plans = []
    for t in range(n_threads):
        small = gen.stress_rows(3, 4099 + t)
        bulk = gen.gradient_rows(3, M + 2047 + 8 * t)
        ar = gen.normal_rows(2, 65536 + 3 + t)
        plans.append({
            "small": (small, [Guarded(small.shape[1], t % 4, small[r]) for r in range(3)],
                      Guarded(small.shape[1], t % 4)),
            "bulk": (bulk, [Guarded(bulk.shape[1], 0, bulk[r]) for r in range(3)],
                     Guarded(bulk.shape[1])),
            "ar": (ar, [Guarded(ar.shape[1], 1, ar[r]) for r in range(2)]),
        })
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(n_threads)

    def worker(p):
        try:
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                for _ in range(iters):
                    for key in ("small", "bulk"):
                        rows, srcs, out = p[key]
                        df.detfold_sum_ptrs(out.t, [x.t for x in srcs], 3, rows.shape[1])
                    rows, arenas = p["ar"]
                    # W=2 with the mean 0.5: the arenas are identical after the
                    # first call, so every later call reproduces the same bits
                    df.detfold_loopback_allreduce([x.t for x in arenas], 2, rows.shape[1], 0.5)
                    # an invalid call from this thread must fail alone, as a status
                    assert df.status_sum_ptrs(out.t, [x.t for x in srcs], 0, 8) == df.STATUS["DETFOLD_ERR_WORLD"]
            s.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(p,)) for p in plans]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a worker did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    for t, p in enumerate(plans):
        for key in ("small", "bulk"):
            rows, srcs, out = p[key]
            assert out.intact()
            assert_bitwise(out.host(), oracle.fold(rows), f"thread {t} {key}")
        rows, arenas = p["ar"]
        want = [rows[r].copy() for r in range(2)]
        oracle.allreduce(want, np.float32(0.5))
        for r in range(2):
            assert arenas[r].intact()
            assert_bitwise(arenas[r].host(), want[r], f"thread {t} all-reduce rank {r}")
    assert df.detfold_pipeline_timeouts() == 0
