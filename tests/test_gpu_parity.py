"""GPU parity: the CUDA library against the CPU oracle, bit for bit (0 ULP).

Fold and mean: mamba-rs 0.6.2 src/dist/reducer.rs (module doc,
`reduce_sum_reference`, `LoopbackWorld::run_round`). Gate patterns: memra-engine
0.128.0 tests/tp_ar_gpu.rs (sizes 1..65536, repeat call gives 2S, red arm) and
memra-engine 0.136.0 tests/gdn_packed_gpu.rs (graph replay with rebinding).
Every device buffer has sentinel guard bands that must survive each call.
"""
import numpy as np
import pytest
import torch

import detfold_inputs as gen
import oracle
from gpu_util import Guarded, assert_bitwise, nonvacuous

import deterministic_fixed_order_gb300 as df

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

C1_SIZES = [1, 4, 1024, 4096, 16384, 65536]
C5_LEN = (1 << 20) + 7


def sync():
    torch.cuda.synchronize()


def run_stacked(rows: np.ndarray, offset: int = 0, out_offset: int | None = None):
    W, n = rows.shape
    st = Guarded(W * n, offset, rows)
    out = Guarded(n, offset if out_offset is None else out_offset)
    df.detfold_sum_stacked(out.t, st.t, W, n)
    sync()
    assert st.intact() and out.intact(), "guard band overwritten"
    return out.host()


def run_ptrs(rows: np.ndarray, offsets=None, out_offset: int = 0):
    W, n = rows.shape
    offsets = offsets or [0] * W
    srcs = [Guarded(n, offsets[r], rows[r]) for r in range(W)]
    out = Guarded(n, out_offset)
    df.detfold_sum_ptrs(out.t, [s.t for s in srcs], W, n)
    sync()
    assert all(s.intact() for s in srcs) and out.intact(), "guard band overwritten"
    for r in range(W):
        assert_bitwise(srcs[r].host(), rows[r], f"source {r} modified")
    return out.host()


def run_allreduce(rows: np.ndarray, scale: float = 1.0, offsets=None, staged_flags=None):
    W, n = rows.shape
    offsets = offsets or [0] * W
    arenas = [Guarded(n, offsets[r], rows[r]) for r in range(W)]
    if staged_flags is None:
        df.detfold_loopback_allreduce([a.t for a in arenas], W, n, scale)
    else:
        nb = df.detfold_staged_workspace_bytes(n, W)
        ws = torch.empty(max(1, nb // 4), dtype=torch.float32, device="cuda")
        if staged_flags == 0:  # the plain call of the C ABI
            df.detfold_loopback_allreduce_staged([a.t for a in arenas], W, n, scale, ws, nb)
        else:
            df.detfold_loopback_allreduce_staged_ex([a.t for a in arenas], W, n, scale, staged_flags,
                                                    ws, nb)
    sync()
    assert all(a.intact() for a in arenas), "guard band overwritten"
    return [a.host() for a in arenas]


def oracle_allreduce(rows: np.ndarray, scale: float = 1.0):
    arenas = [rows[r].copy() for r in range(rows.shape[0])]
    oracle.allreduce(arenas, np.float32(scale))
    return arenas


# ------------------------------------------------------------------ C1: W = 2 decode-join sizes

@pytest.mark.parametrize("n", C1_SIZES)
def test_c1_stacked_bitwise_and_repeat_call(n):
    rows = gen.c1_rows(2, n)
    want = oracle.fold_stacked(rows)
    got = run_stacked(rows)
    assert_bitwise(got, want, f"C1 n={n}")
    nz, am = nonvacuous(got)
    assert nz > 0 and am > 0
    # Repeat call: both rows now hold S (as after an all-reduce): exactly 2S.
    again = run_stacked(np.stack([got, got]))
    assert_bitwise(again, oracle.fold(np.stack([want, want])), f"C1 repeat n={n}")
    assert np.array_equal(again.astype(np.float64), 2.0 * want.astype(np.float64))


@pytest.mark.parametrize("n", C1_SIZES)
def test_c1_ptrs_and_allreduce_forms(n):
    rows = gen.c1_rows(2, n)
    want = oracle.fold(rows)
    assert_bitwise(run_ptrs(rows), want, f"C1 ptrs n={n}")
    arenas = [Guarded(n, 0, rows[r]) for r in range(2)]
    for call in range(2):
        df.detfold_loopback_allreduce([a.t for a in arenas], 2, n, 1.0)
        sync()
        exp = want if call == 0 else oracle.fold(np.stack([want, want]))
        for r in range(2):
            assert_bitwise(arenas[r].host(), exp, f"C1 all-reduce n={n} call={call} rank={r}")
        assert all(a.intact() for a in arenas)


def test_red_arm_fold_without_peer_contribution_diverges():
    # In-place fold with a zero stage: rank 0 keeps its own partial, which
    # must not reproduce the sum (else the bitwise gate proves nothing).
    n = 4096
    a, b = gen.vecf(n, 5), gen.vecf(n, 6)
    dst = Guarded(n, 0, a)
    stage = Guarded(n, 0, np.zeros(n, np.float32))
    df.detfold_sum_ptrs(dst.t, [dst.t, stage.t], 2, n)
    sync()
    got = dst.host()
    want = oracle.fold(np.stack([a, b]))
    same = int(np.count_nonzero(got.view(np.uint32) == want.view(np.uint32)))
    assert same < n
    assert_bitwise(got, a, "fold with zero stage")


# ------------------------------------------------------------------ heads, tails, phases

@pytest.mark.parametrize("W", [1, 2, 3, 5, 8])
def test_every_small_length_and_head_offset(W):
    rows_all = gen.stress_rows(W, 64)
    for n in range(1, 65):
        rows = np.ascontiguousarray(rows_all[:, :n])
        want = oracle.fold(rows)
        for off in range(8):
            assert_bitwise(run_ptrs(rows, [off] * W, off), want, f"ptrs W={W} n={n} off={off}")
        for off in (0, 1, 3, 5):
            assert_bitwise(run_stacked(rows, off), want, f"stacked W={W} n={n} off={off}")


@pytest.mark.parametrize("W", [2, 3, 4, 6, 7, 8, 9, 16])
@pytest.mark.parametrize("n", [1, 7, 1000, 4099, C5_LEN])
def test_mismatched_phases(W, n):
    rows = gen.stress_rows(W, n)
    want = oracle.fold(rows)
    offs = [(r * 3) % 8 for r in range(W)]
    assert_bitwise(run_ptrs(rows, offs, out_offset=5), want, f"ptrs W={W} n={n}")
    got = run_allreduce(rows, float(oracle.mean_scale(W)), offs)
    exp = oracle_allreduce(rows, oracle.mean_scale(W))
    for r in range(W):
        assert_bitwise(got[r], exp[r], f"all-reduce W={W} n={n} rank={r}")


@pytest.mark.parametrize("W", [2, 3, 5, 8])
def test_mixed_phase_allreduce_across_pass_edges(W):
    # The realigned all-reduce folds 31 logical vectors (248 elements) per
    # warp pass and stores each arena's aligned vectors whole inside a pass,
    # element by element at its two ends. Lengths on both sides of several
    # pass edges, with random per-arena phases, must still give every arena
    # the oracle's bits, and leave the guard bands intact.
    rng = np.random.default_rng(7 + W)
    lengths = sorted({*range(1, 40), *(8 * k + d for k in (31, 62, 93, 155) for d in (-9, -1, 0, 1, 7, 9, 17)),
                      2047, 4099, 8 * 31 * 64 + 5})
    for n in lengths:
        rows = gen.stress_rows(W, n, seed0=int(rng.integers(1, 1 << 30)))
        offs = [int(x) for x in rng.integers(0, 8, size=W)]
        scale = float(oracle.mean_scale(W)) if n % 2 else 1.0
        got = run_allreduce(rows, scale, offs)
        exp = oracle_allreduce(rows, np.float32(scale))
        for r in range(W):
            assert_bitwise(got[r], exp[r], f"mixed-phase all-reduce W={W} n={n} offs={offs} rank={r}")


# ------------------------------------------------------------------ C5: odd worlds, stress values

@pytest.mark.parametrize("W", [3, 6])
@pytest.mark.parametrize("variant", ["base+4", "per-rank-phase"])
def test_c5_stress_sum_mean_and_allreduce(W, variant):
    rows = gen.stress_rows(W, C5_LEN)
    s_want = oracle.fold(rows)
    m = oracle.mean_scale(W)
    mean_want = oracle.scale(s_want, m)
    offs = [1] * W if variant == "base+4" else [r % 4 for r in range(W)]
    if variant == "base+4":
        assert_bitwise(run_stacked(rows, 1, 1), s_want, f"C5 stacked W={W}")
    got = run_ptrs(rows, offs, out_offset=1)
    assert_bitwise(got, s_want, f"C5 ptrs W={W} {variant}")
    # the mean as its own pass over the sum
    buf = Guarded(C5_LEN, 1, got)
    df.detfold_scale(buf.t, C5_LEN, float(m))
    sync()
    assert buf.intact()
    assert_bitwise(buf.host(), mean_want, f"C5 mean W={W}")
    # fused all-reduce with the mean in registers, and the staged comparator
    for flags in (None, 0, 1, 2, 3, 4):
        ar = run_allreduce(rows, float(m), offs, staged_flags=flags)
        for r in range(W):
            assert_bitwise(ar[r], mean_want, f"C5 all-reduce W={W} flags={flags} rank={r}")
    nz, am = nonvacuous(s_want)
    assert nz > 0 and am > 0


def test_c5_special_columns():
    # Elements 0..15 of the stress rows hold signed-zero, subnormal,
    # cancellation and order-sensitive columns (see detfold_inputs/gen.c).
    for W in (3, 6):
        rows = np.ascontiguousarray(gen.stress_rows(W, 64)[:, :16])
        want = oracle.fold(rows)
        assert_bitwise(run_ptrs(rows), want, f"specials W={W}")
        assert want.view(np.uint32)[0] == 0x80000000  # all -0 stays -0


# ------------------------------------------------------------------ runtime-W kernels

@pytest.mark.parametrize("W", [9, 16, 33, 256])
@pytest.mark.parametrize("n", [1, 1000, 4099, (1 << 17) + 3])
def test_generic_world_sizes(W, n):
    rows = gen.normal_rows(W, n)
    want = oracle.fold(rows)
    assert_bitwise(run_stacked(rows), want, f"generic stacked W={W} n={n}")
    assert_bitwise(run_ptrs(rows), want, f"generic ptrs W={W} n={n}")
    got = run_allreduce(rows, 0.5)
    exp = oracle_allreduce(rows, 0.5)
    for r in (0, W - 1):
        assert_bitwise(got[r], exp[r], f"generic all-reduce W={W} n={n}")


@pytest.mark.parametrize("W", [2, 4, 8])
@pytest.mark.parametrize("k", ["first", "last"])
@pytest.mark.parametrize("n", [4099, C5_LEN])
def test_in_place_fold(W, k, n):
    rows = gen.gradient_rows(W, n)
    want = oracle.fold(rows)
    srcs = [Guarded(n, 0, rows[r]) for r in range(W)]
    kk = 0 if k == "first" else W - 1
    df.detfold_sum_ptrs(srcs[kk].t, [s.t for s in srcs], W, n)
    sync()
    assert all(s.intact() for s in srcs)
    assert_bitwise(srcs[kk].host(), want, f"in place W={W} k={k}")


@pytest.mark.parametrize("W", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [1, 9, 1034, 4099, 16391, 1 << 17, (1 << 17) + 1])
@pytest.mark.parametrize("off", [0, 1, 4, 7])
def test_small_path_modes_with_heads_and_tails(W, n, off):
    # Every mode of the small-payload launch (n <= 2^17 elements) with a head
    # and a tail: the read-only sum, the in-place sum, and the fused
    # all-reduce with the mean; n = 2^17 + 1 is the first bandwidth-path length.
    # 1034 at offset 1 (head 7, 128 vectors, tail 3) and 16391 at offset 1
    # (head 7, 2048 vectors) give grids of exactly one thread per vector.
    rows = gen.stress_rows(W, n)
    want = oracle.fold(rows)
    assert_bitwise(run_ptrs(rows, [off] * W, off), want, f"sum W={W} n={n} off={off}")
    srcs = [Guarded(n, off, rows[r]) for r in range(W)]
    df.detfold_sum_ptrs(srcs[W - 1].t, [t.t for t in srcs], W, n)
    sync()
    assert all(t.intact() for t in srcs)
    assert_bitwise(srcs[W - 1].host(), want, f"in place W={W} n={n} off={off}")
    scale = float(oracle.mean_scale(W))
    got = run_allreduce(rows, scale, [off] * W)
    exp = oracle_allreduce(rows, scale)
    for r in range(W):
        assert_bitwise(got[r], exp[r], f"all-reduce W={W} n={n} off={off} r={r}")


@pytest.mark.parametrize("W", [2, 3, 8])
@pytest.mark.parametrize("n,off", [(1028, 3), (1028, 0), (4096, 0), (4100, 1), (65536, 0)])
def test_small_path_stacked_exact_and_ragged_grids(W, n, off):
    # Stacked rows of n = 4 (mod 8) elements sit at alternating 32-byte phases,
    # so the call takes 16-byte vectors: (1028, 3) has head 1, 256 vectors
    # (an exact grid) and tail 3; (1028, 0) has 257 vectors (ragged grid).
    rows = gen.stress_rows(W, n)
    assert_bitwise(run_stacked(rows, off), oracle.fold(rows), f"stacked W={W} n={n} off={off}")


# ------------------------------------------------------------------ all-reduce: fused vs staged

@pytest.mark.parametrize("W", [1, 2, 3, 4, 6, 8])
@pytest.mark.parametrize("n", [1, 5, 7, 4099, 100_003])
def test_allreduce_fused_and_staged_match_oracle(W, n):
    rows = gen.normal_rows(W, n)
    for scale in (1.0, float(oracle.mean_scale(W))):
        exp = oracle_allreduce(rows, scale)
        for flags in (None, 0, 1, 2, 3, 4, 7):
            got = run_allreduce(rows, scale, staged_flags=flags)
            for r in range(W):
                assert_bitwise(got[r], exp[r], f"W={W} n={n} scale={scale} flags={flags} r={r}")


def test_allreduce_repeat_call_matches_oracle_on_updated_state():
    n = 65536 + 3
    for W in (2, 4, 6):
        rows = gen.normal_rows(W, n)
        arenas = [Guarded(n, 0, rows[r]) for r in range(W)]
        host = [rows[r].copy() for r in range(W)]
        for call in range(3):
            df.detfold_loopback_allreduce([a.t for a in arenas], W, n, 1.0)
            oracle.allreduce(host)
            sync()
            for r in range(W):
                assert_bitwise(arenas[r].host(), host[r], f"W={W} call={call} rank={r}")


def test_len_zero_and_one_rank_are_noops():
    a = Guarded(16, 0, np.arange(16, dtype=np.float32))
    df.detfold_loopback_allreduce([a.t], 1, 16, 1.0)
    df.detfold_sum_ptrs(a.t, [a.t], 1, 16)
    df.detfold_scale(a.t, 16, 1.0)
    df.detfold_loopback_allreduce([a.t], 1, 0, 0.5)
    sync()
    assert_bitwise(a.host(), np.arange(16, dtype=np.float32), "no-op calls changed data")
    assert a.intact()


# ------------------------------------------------------------------ pure movement

def _random_bits(n, seed):
    # every 32-bit pattern is fair game for movement: NaN payloads, -0, subnormals
    return np.random.default_rng(seed).integers(0, 2 ** 32, size=n, dtype=np.uint64) \
        .astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("span", [1, 1024, 16384, (1 << 20) + 3])
@pytest.mark.parametrize("W", [2, 3, 8])
def test_broadcast_and_all_gather_move_bytes_exactly(span, W):
    # broadcast: the root's buffer lands on every other rank byte for byte
    src_h = _random_bits(span, 31 + span)
    src = Guarded(span, 3, src_h)
    dsts = [Guarded(span, 3 if r % 2 else 0) for r in range(W - 1)]
    df.detfold_broadcast([d.t for d in dsts], W - 1, src.t, span)
    sync()
    for k, d in enumerate(dsts):
        assert_bitwise(d.host(), src_h, f"broadcast span={span} dst={k}")
        assert d.intact()
    assert src.intact()
    assert_bitwise(src.host(), src_h, "broadcast source modified")
    # all-gather: rank-order concatenation, identical on every rank
    parts_h = [_random_bits(span, 41 + r + span) for r in range(W)]
    parts = [Guarded(span, r % 2, parts_h[r]) for r in range(W)]
    outs = [Guarded(W * span, (r * 5) % 8) for r in range(W)]
    df.detfold_all_gather([o.t for o in outs], W, [p.t for p in parts], span)
    sync()
    want = np.concatenate(parts_h)
    for r, o in enumerate(outs):
        assert_bitwise(o.host(), want, f"all-gather span={span} rank={r}")
        assert o.intact()


@pytest.mark.parametrize("span", [1, 7, 1024, 4099, 16384, 1 << 17, (1 << 17) + 1])
@pytest.mark.parametrize("W", [2, 3, 8, 12])
@pytest.mark.parametrize("off", [0, 1, 4, 7])
def test_movement_at_one_phase_with_heads_and_tails(span, W, off):
    # Every pointer at one phase: the vector movement kernels, with a head and
    # a tail at offsets 1 and 7; spans up to 2^17 take the small-move kernel
    # (one pair-vector per thread), 2^17 + 1 the looping kernel. W = 12 parts
    # is past the one-launch all-gather (at most 8 parts): one launch per part.
    src_h = _random_bits(span, 57 + span)
    src = Guarded(span, off, src_h)
    dsts = [Guarded(span, off) for _ in range(W - 1)]
    df.detfold_broadcast([d.t for d in dsts], W - 1, src.t, span)
    sync()
    for k, d in enumerate(dsts):
        assert d.intact()
        assert_bitwise(d.host(), src_h, f"broadcast span={span} off={off} dst={k}")
    parts_h = [_random_bits(span, 67 + r + span) for r in range(W)]
    parts = [Guarded(span, off, parts_h[r]) for r in range(W)]
    outs = [Guarded(W * span, off) for _ in range(W)]
    df.detfold_all_gather([o.t for o in outs], W, [p.t for p in parts], span)
    sync()
    want = np.concatenate(parts_h)
    for r, o in enumerate(outs):
        assert o.intact()
        assert_bitwise(o.host(), want, f"all-gather span={span} off={off} rank={r}")


@pytest.mark.parametrize("layout", ["mixed", "aligned", "aligned+head"])
def test_broadcast_many_destinations_splits_launches(layout):
    # more destinations than one parameter block holds (250 pairs per launch):
    # mixed phases take the scalar kernel, one phase the small-move kernel
    span, nd = (1003 if layout == "aligned+head" else 1000), 256
    src_h = _random_bits(span, 7)
    off = {"mixed": 0, "aligned": 0, "aligned+head": 1}[layout]
    src = Guarded(span, off, src_h)
    dsts = [Guarded(span, r % 8 if layout == "mixed" else off) for r in range(nd)]
    df.detfold_broadcast([d.t for d in dsts], nd, src.t, span)
    sync()
    for d in dsts:
        assert_bitwise(d.host(), src_h, "broadcast to 256")
        assert d.intact()


# ------------------------------------------------------------------ C2: small payload + graphs

@pytest.mark.parametrize("n", [4096, 65536])
def test_c2_small_path_and_graph_replay(n):
    rows = gen.c1_rows(2, n)
    want = oracle.fold(rows)
    st = Guarded(2 * n, 0, rows)
    out = Guarded(n)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        df.detfold_sum_stacked(out.t, st.t, 2, n)  # warm up outside capture
    stream.synchronize()
    out.t.zero_()
    sync()
    with torch.cuda.graph(g, stream=stream):  # C2: 10,000 back-to-back folds in one graph
        for _ in range(10_000):
            df.detfold_sum_stacked(out.t, st.t, 2, n)
    for _ in range(3):
        g.replay()
    sync()
    assert out.intact() and st.intact()
    assert_bitwise(out.host(), want, f"graph replay n={n}")


def test_graph_recapture_with_rebound_buffers():
    # The pointer table is baked in at capture: a second capture over new
    # buffers (the canonical/alternate swap of the graph-rebind gate) must
    # give the same bits on its own inputs.
    n = 4096
    rows = gen.c1_rows(2, n)
    want = oracle.fold(rows)
    bufs = [(Guarded(n, 0, rows[0]), Guarded(n, 0, rows[1]), Guarded(n)) for _ in range(2)]
    graphs = []
    stream = torch.cuda.Stream()
    for a, b, o in bufs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(50):
                df.detfold_sum_ptrs(o.t, [a.t, b.t], 2, n)
        graphs.append(g)
    for order in ((0, 1), (1, 0)):
        for k in order:
            bufs[k][2].t.zero_()
            graphs[k].replay()
        sync()
        for a, b, o in bufs:
            assert_bitwise(o.host(), want, "recaptured graph")
            assert o.intact()


def test_many_back_to_back_small_folds_on_a_stream():
    n = 4096
    rows = gen.c1_rows(2, n)
    want = oracle.fold(rows)
    st = Guarded(2 * n, 0, rows)
    out = Guarded(n)
    for _ in range(2000):
        df.detfold_sum_stacked(out.t, st.t, 2, n)
    sync()
    assert_bitwise(out.host(), want, "2000 back-to-back folds")


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.slow
def test_c3_full_size_w8_gradient_bitwise():
    W, n = 8, 1 << 26
    rows = gen.gradient_rows(W, n)
    want = oracle.fold_stacked(rows)
    st = torch.from_numpy(rows).cuda()
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    df.detfold_sum_stacked(out, st, W, n)
    sync()
    assert_bitwise(out.cpu().numpy(), want, "C3 stacked")
    out.zero_()
    df.detfold_sum_ptrs(out, [st[r] for r in range(W)], W, n)
    sync()
    assert_bitwise(out.cpu().numpy(), want, "C3 ptrs")
    nz, am = nonvacuous(want)
    assert nz > 0.99 * n and am > 1.0


@pytest.mark.slow
def test_c4_full_size_w4_fused_and_staged_bitwise():
    W, n = 4, 100_000_000
    rows = gen.normal_rows(W, n)
    exp = oracle_allreduce(rows, 0.25)
    fused = [torch.from_numpy(rows[r]).cuda() for r in range(W)]
    df.detfold_loopback_allreduce(fused, W, n, 0.25)
    sync()
    for r in range(W):
        assert_bitwise(fused[r].cpu().numpy(), exp[r], f"C4 fused rank {r}")
    del fused
    nb = df.detfold_staged_workspace_bytes(n, W)
    ws = torch.empty(nb // 4, dtype=torch.float32, device="cuda")
    for flags in (0, df.DETFOLD_STAGED_SEPARATE_SCALE | df.DETFOLD_STAGED_REVERSE_DELIVERY,
                  df.DETFOLD_STAGED_CE_COPIES):
        staged = [torch.from_numpy(rows[r]).cuda() for r in range(W)]
        if flags == 0:
            df.detfold_loopback_allreduce_staged(staged, W, n, 0.25, ws, nb)
        else:
            df.detfold_loopback_allreduce_staged_ex(staged, W, n, 0.25, flags, ws, nb)
        sync()
        for r in range(W):
            assert_bitwise(staged[r].cpu().numpy(), exp[r], f"C4 staged flags={flags} rank {r}")
        del staged


# ------------------------------------------------------------------ degenerate and extreme inputs

def _nonfinite_rows(W, n, seed):
    rows = gen.normal_rows(W, n)
    rng = np.random.default_rng(seed)
    specials = np.array([np.inf, -np.inf, np.nan], dtype=np.float32)
    for r in range(W):
        pick = rng.random(n) < 0.02
        rows[r, pick] = specials[rng.integers(0, 3, size=int(pick.sum()))]
    return rows


@pytest.mark.parametrize("W", [2, 3, 8])
@pytest.mark.parametrize("n", [4099, (1 << 20) + 7])
def test_nonfinite_inputs_match_by_class(W, n):
    # Inf and NaN propagate through the chain on both sides. Finite and
    # infinite results must match bitwise; NaN results must be NaN on both
    # sides (a GPU returns a canonical NaN, a host may keep an input payload).
    rows = _nonfinite_rows(W, n, 17 + W)
    want = oracle.fold(rows)
    for got in (run_stacked(rows), run_ptrs(rows), run_allreduce(rows)[W - 1]):
        nan_w, nan_g = np.isnan(want), np.isnan(got)
        assert np.array_equal(nan_w, nan_g), "NaN positions differ"
        assert_bitwise(got[~nan_g], want[~nan_w], f"non-NaN words W={W} n={n}")
        assert nan_w.sum() > 0 and np.isinf(want).sum() > 0


@pytest.mark.slow
def test_lengths_beyond_int32():
    # 64-bit element indexing: the reference's kernel ABI stops at i32 lengths.
    n = (1 << 31) + 77
    rows = gen.c1_rows(2, n)                       # 17.2 GB of host data
    d = torch.from_numpy(rows).cuda()
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    df.detfold_sum_stacked(out, d, 2, n)
    torch.cuda.synchronize()
    idx = np.unique(np.r_[np.arange(0, 64), np.arange((1 << 31) - 64, (1 << 31) + 64),
                          np.arange(n - 64, n),
                          np.random.default_rng(5).integers(0, n, 4096)])
    want = oracle.fold(np.ascontiguousarray(rows[:, idx]))
    got = out[torch.from_numpy(idx).cuda()].cpu().numpy()
    assert_bitwise(got, want, "len > 2^31 stacked")
    # the fused all-reduce in place, on the same data
    arenas = [d[0], d[1]]
    df.detfold_loopback_allreduce(arenas, 2, n, 0.5)
    torch.cuda.synchronize()
    want_ar = oracle.scale(want, np.float32(0.5))
    ti = torch.from_numpy(idx).cuda()
    for r in range(2):
        assert_bitwise(arenas[r][ti].cpu().numpy(), want_ar, f"len > 2^31 all-reduce rank {r}")
    assert df.detfold_pipeline_timeouts() == 0


# ------------------------------------------------------------------ latency-floor probes

@pytest.mark.parametrize("pdl", [0, 1])
def test_floor_probes(pdl):
    # The probes a graph of small folds is compared against (their own
    # library): the empty kernel runs, and the one-warp round trip copies
    # exactly 32 floats.
    import bench
    probes = bench.Probes()
    src = Guarded(32, 0, np.arange(1, 33, dtype=np.float32))
    dst = Guarded(32)
    probes.launch_floor(5, pdl)
    probes.memory_floor(src.t, dst.t, 5, pdl)
    sync()
    assert dst.intact() and src.intact()
    assert_bitwise(dst.host(), np.arange(1, 33, dtype=np.float32), "memory floor copy")
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    dst.t.zero_()
    sync()
    with torch.cuda.graph(g, stream=stream):
        probes.launch_floor(20, pdl, stream)
        probes.memory_floor(src.t, dst.t, 20, pdl, stream)
    g.replay()
    sync()
    assert dst.intact()
    assert_bitwise(dst.host(), np.arange(1, 33, dtype=np.float32), "memory floor copy in a graph")


@pytest.mark.parametrize("n", [1024, 4096, 65536, 1 << 17])
def test_same_shape_floor_probe_moves_the_fold_bytes(n):
    # the same-launch-shape floor of the small W=2 fold reads both sources
    # and writes n floats: even elements from src0, odd ones from src1
    import bench
    probes = bench.Probes()
    rows = gen.c1_rows(2, n)
    s0 = Guarded(n, 0, rows[0])
    s1 = Guarded(n, 0, rows[1])
    out = Guarded(n)
    probes.same_shape_floor(out.t, s0.t, s1.t, n, 3)
    sync()
    want = rows[0].copy()
    want[1::2] = rows[1][1::2]
    assert out.intact() and s0.intact() and s1.intact()
    assert_bitwise(out.host(), want, f"same-shape probe n={n}")


def test_binding_enqueues_on_torchs_current_stream():
    # the binding's fast query of torch's current stream agrees with torch's
    # public one, inside and outside a stream context, and in another thread
    assert df._stream(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert df._stream(None) == s.cuda_stream == torch.cuda.current_stream().cuda_stream
    assert df._stream(None) == torch.cuda.current_stream().cuda_stream
    import threading
    seen = []

    def other():
        t = torch.cuda.Stream()
        with torch.cuda.stream(t):
            seen.append(df._stream(None) == t.cuda_stream)
        seen.append(df._stream(None) == torch.cuda.current_stream().cuda_stream)

    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert seen == [True, True]
