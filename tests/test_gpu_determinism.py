"""Determinism arm: every entry point, K runs on identical inputs, 0 words differ.

After memra-engine 0.123.0 src/bin/moe_tp2_repro.rs (determinism arm, with
its non-degeneracy guard) and the fixed-order contract of mamba-rs 0.6.2
src/dist/reducer.rs (the bits do not depend on schedule, transport or
delivery order): each call runs 8 times, serially and concurrently on four
streams, and the different entry points agree with each other bit for bit.
"""
import numpy as np
import pytest
import torch

import detfold_inputs as gen
import oracle
from gpu_util import Guarded, assert_bitwise

import deterministic_fixed_order_gb300 as df
from deterministic_fixed_order_gb300.determinism import determinism_diff

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

N = (1 << 22) + 5


def _ok(rep, what):
    assert rep["verdict"] == "DETERMINISTIC", (what, rep)
    assert rep["nonzero"] > 0.9 * rep["words"], (what, rep)


def test_every_entry_point_is_deterministic():
    W = 6
    rows = gen.stress_rows(W, N)
    st = torch.from_numpy(rows).cuda()
    out = torch.empty(N, device="cuda")
    _ok(determinism_diff(lambda k: df.detfold_sum_stacked(out, st, W, N), lambda k: out),
        "sum_stacked")
    offs = [Guarded(N, r % 4, rows[r]) for r in range(W)]
    out2 = Guarded(N, 3)
    _ok(determinism_diff(lambda k: df.detfold_sum_ptrs(out2.t, [o.t for o in offs], W, N),
                         lambda k: out2.t), "sum_ptrs mismatched phases")
    table = df.device_table([o.t for o in offs])
    _ok(determinism_diff(lambda k: df.detfold_sum_ptrs_dev(out2.t, table, W, N),
                         lambda k: out2.t), "sum_ptrs_dev")
    arenas = [torch.empty(N, device="cuda") for _ in range(W)]
    src = [torch.from_numpy(rows[r]).cuda() for r in range(W)]

    def reset(k):
        for a, s in zip(arenas, src):
            a.copy_(s)
    scale = float(oracle.mean_scale(W))
    _ok(determinism_diff(lambda k: df.detfold_loopback_allreduce(arenas, W, N, scale),
                         lambda k: arenas, reset), "fused all-reduce")
    # arenas at different 16-byte phases (the bulk pipeline with per-arena
    # offsets at this length)
    mixed = [Guarded(N, (3 * r) % 8, rows[r]) for r in range(W)]

    def reset_mixed(k):
        for m, s in zip(mixed, src):
            m.t.copy_(s)
    _ok(determinism_diff(lambda k: df.detfold_loopback_allreduce([m.t for m in mixed], W, N, scale),
                         lambda k: [m.t for m in mixed], reset_mixed), "fused all-reduce, mixed phases")
    nb = df.detfold_staged_workspace_bytes(N, W)
    ws = torch.empty(nb // 4, device="cuda")
    for flags in (0, 1, 4, 7):
        _ok(determinism_diff(
            lambda k: df.detfold_loopback_allreduce_staged_ex(arenas, W, N, scale, flags, ws, nb),
            lambda k: arenas, reset), f"staged flags={flags}")
    n2 = 4096
    c2 = torch.from_numpy(gen.c1_rows(2, n2)).cuda()
    o2 = torch.empty(n2, device="cuda")
    _ok(determinism_diff(lambda k: df.detfold_sum_stacked(o2, c2, 2, n2), lambda k: o2,
                         repeats=32), "small path")
    dsts = [torch.empty(N, device="cuda") for _ in range(3)]
    _ok(determinism_diff(lambda k: df.detfold_broadcast(dsts, 3, src[0], N), lambda k: dsts),
        "broadcast")
    outs = [torch.empty(W * 1000, device="cuda") for _ in range(W)]
    parts = [s[:1000] for s in src]
    _ok(determinism_diff(lambda k: df.detfold_all_gather(outs, W, parts, 1000), lambda k: outs),
        "all_gather")


def test_concurrent_runs_on_four_streams_agree():
    W = 8
    rows = gen.gradient_rows(W, N)
    st = torch.from_numpy(rows).cuda()
    outs = [torch.empty(N, device="cuda") for _ in range(8)]
    streams = [torch.cuda.Stream() for _ in range(4)]
    torch.cuda.synchronize()
    rep = determinism_diff(lambda k: df.detfold_sum_stacked(outs[k], st, W, N),
                           lambda k: outs[k], repeats=8, streams=streams)
    _ok(rep, "concurrent sum_stacked")
    assert_bitwise(outs[0].cpu().numpy(), oracle.fold_stacked(rows), "concurrent vs oracle")


def test_entry_points_agree_with_each_other():
    # The same addends through every route: stacked, pointer table at any
    # phase, device table, fused all-reduce, staged (SM and copy-engine
    # movement, either delivery order) -- one set of bits.
    W = 5
    rows = gen.stress_rows(W, N)
    want = oracle.fold(rows)
    got = {}
    st = torch.from_numpy(rows).cuda()
    out = torch.empty(N, device="cuda")
    df.detfold_sum_stacked(out, st, W, N)
    got["stacked"] = out.cpu().numpy()
    srcs = [Guarded(N, (2 * r) % 8, rows[r]) for r in range(W)]
    o = Guarded(N, 1)
    df.detfold_sum_ptrs(o.t, [s.t for s in srcs], W, N)
    got["ptrs"] = o.host()
    df.detfold_sum_ptrs_dev(o.t, df.device_table([s.t for s in srcs]), W, N)
    got["ptrs_dev"] = o.host()
    nb = df.detfold_staged_workspace_bytes(N, W)
    ws = torch.empty(nb // 4, device="cuda")
    for name, flags in (("fused", None), ("staged", 0), ("staged_ce_rev", 5)):
        arenas = [torch.from_numpy(rows[r]).cuda() for r in range(W)]
        if flags is None:
            df.detfold_loopback_allreduce(arenas, W, N, 1.0)
        else:
            df.detfold_loopback_allreduce_staged_ex(arenas, W, N, 1.0, flags, ws, nb)
        got[name] = arenas[W - 1].cpu().numpy()
    torch.cuda.synchronize()
    for name, g in got.items():
        assert_bitwise(g, want, f"route {name}")
