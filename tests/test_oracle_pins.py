"""Pins for the CPU oracle: each expectation here comes from outside the oracle.

Fold and mean: mamba-rs 0.6.2 src/dist/reducer.rs (module doc,
`reduce_sum_reference`). Test data: memra-engine 0.128.0 tests/tp_ar_gpu.rs
(`vecf`, the bitwise host-sum gate, its repeat call and its red arm).
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import detfold_inputs as gen
import ieee_model as M
import oracle
from pins import (MUTANTS, as_bits, bits_array, double_simulated_fold, fold_pin_failures,
                  load_hand_cases, model_fold)


# ---------------------------------------------------------------- the model itself

def test_model_rounding_known_values():
    # ties to even at 1 + 2^-24 and 1 + 3*2^-24
    assert M.round_to_bits(1 + Fraction(1, 2 ** 24)) == 0x3F800000
    assert M.round_to_bits(1 + Fraction(3, 2 ** 24)) == 0x3F800002
    # subnormal quantum, underflow to zero, smallest normal
    assert M.round_to_bits(Fraction(1, 2 ** 149)) == 0x00000001
    assert M.round_to_bits(Fraction(1, 2 ** 150)) == 0x00000000          # tie -> even (0)
    assert M.round_to_bits(Fraction(3, 2 ** 151)) == 0x00000001
    assert M.round_to_bits(Fraction(1, 2 ** 126)) == 0x00800000
    # overflow
    big = Fraction(2 ** 128)
    assert M.round_to_bits(big) == M.POS_INF
    assert M.round_to_bits(-big) == M.NEG_INF
    assert M.round_to_bits(Fraction((1 << 24) - 1) * 2 ** 104) == 0x7F7FFFFF
    # decode/round round-trips every pattern class
    for b in (0x00000001, 0x007FFFFF, 0x00800000, 0x3F800000, 0x7F7FFFFF, 0x80000001, 0xC0490FDB):
        assert M.round_to_bits(M.decode(b)) == b


def test_model_matches_ieee_hardware_add():
    # numpy float32 addition is IEEE round-to-nearest-even without FTZ on
    # x86-64 and aarch64; agreement on random pairs checks the model itself.
    rows = gen.stress_rows(2, 3000)
    a, b = as_bits(rows[0]), as_bits(rows[1])
    hw = as_bits(rows[0] + rows[1])
    for i in range(3000):
        assert M.add(int(a[i]), int(b[i])) == int(hw[i]), i


def test_golden_cases_agree_with_model():
    for name, W, adds, want_sum, want_mean in load_hand_cases():
        s = M.chain(adds)
        assert s == want_sum, name
        if want_mean is not None:
            assert M.mul(s, M.recip(W)) == want_mean, name


# ---------------------------------------------------------------- the fold

def test_oracle_fold_passes_every_pin():
    assert fold_pin_failures(oracle.fold) == []


def test_oracle_fold_stacked_passes_every_pin():
    assert fold_pin_failures(oracle.fold_stacked) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mutant_fails_a_pin(name):
    fails = fold_pin_failures(MUTANTS[name])
    assert fails, f"mutant {name} slipped through every pin"


def test_order_matters_by_brute_force():
    # Every rank order of small order-sensitive columns, through the exact
    # model: the oracle matches the ascending order, and some other order
    # gives different bits (so ascending order is a real constraint).
    cases = load_hand_cases()
    sensitive = 0
    for name, W, adds, _, _ in cases:
        want = M.chain(adds)
        got = int(as_bits(oracle.fold(bits_array(adds).reshape(W, 1)))[0])
        assert got == want, name
        others = {M.chain([adds[p] for p in perm]) for perm in itertools.permutations(range(W))}
        if len(others) > 1:
            sensitive += 1
    assert sensitive >= 3
    rows = gen.stress_rows(5, 256)
    for i in range(0, 256, 17):
        col = [int(x) for x in as_bits(rows[:, i])]
        ascending = M.chain(col)
        assert int(as_bits(oracle.fold(rows[:, i:i + 1]))[0]) == ascending


def test_workload_data_is_order_sensitive_and_nonvacuous():
    # Zero or symmetric data would make any order agree; the recipes must not.
    for recipe, W in (("gradient", 8), ("stress", 3), ("stress", 6), ("normal", 4)):
        rows = gen.recipe_rows(recipe, W, 1 << 15)
        s = oracle.fold(rows)
        assert np.count_nonzero(s) > 0.9 * s.size
        assert np.max(np.abs(s)) > 0
        rev = double_simulated_fold(np.ascontiguousarray(rows[::-1]))
        assert oracle.bit_diffs(s, rev) > 0, recipe


# ---------------------------------------------------------------- the C1 gate

@pytest.mark.parametrize("n", [1, 4, 1024, 4096, 16384, 65536])
def test_w2_vecf_sums_are_exact(n):
    # vecf values are k * 2^-23 with |k| < 2^23, so a + b needs at most 24
    # significant bits: the binary32 sum is the exact sum.
    a = gen.vecf(n, 11 + n)
    b = gen.vecf(n, 77 + n)
    rows = gen.c1_rows(2, n)
    assert np.array_equal(as_bits(rows[0]), as_bits(a))
    assert np.array_equal(as_bits(rows[1]), as_bits(b))
    exact = a.astype(np.float64) + b.astype(np.float64)
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
    s = oracle.fold(rows)
    assert np.array_equal(s.astype(np.float64), exact)
    # The repeat call: both ranks hold S, so the fold gives 2S exactly.
    twice = oracle.fold(np.stack([s, s]))
    assert np.array_equal(twice.astype(np.float64), 2.0 * exact)


def test_red_arm_dropping_a_rank_diverges():
    n = 4096
    rows = np.stack([gen.vecf(n, 5), gen.vecf(n, 6)])
    full = oracle.fold(rows)
    dropped = oracle.fold(np.stack([rows[0], np.zeros(n, np.float32)]))
    same = n - oracle.bit_diffs(full, dropped)
    assert same < n


def test_vecf_matches_the_page_definition():
    # An independent pure-Python restatement of the page's generator.
    def vecf_py(n, seed):
        s = (seed * 0x9E3779B97F4A7C15) & (2 ** 64 - 1) | 1
        out = []
        for _ in range(n):
            s ^= (s << 13) & (2 ** 64 - 1)
            s ^= s >> 7
            s ^= (s << 17) & (2 ** 64 - 1)
            out.append((Fraction(s >> 40, 2 ** 24) - Fraction(1, 2)) * 2)
        return out
    for seed in (15, 81, 5, 6):
        want = vecf_py(300, seed)
        got = gen.vecf(300, seed)
        assert [Fraction(float(x)) for x in got] == want


# ---------------------------------------------------------------- mean

def test_mean_scale_is_rounded_reciprocal():
    for W in range(1, 300):
        assert M.bits_of(float(oracle.mean_scale(W))) == M.recip(W), W


def test_golden_means():
    for name, W, adds, _, want in load_hand_cases():
        if want is None:
            continue
        s = oracle.fold(bits_array(adds).reshape(W, 1))
        m = oracle.scale(s, oracle.mean_scale(W))
        assert int(as_bits(m)[0]) == want, name


@pytest.mark.parametrize("W", [3, 4, 6, 8])
def test_mean_matches_exact_model(W):
    rows = gen.stress_rows(W, 400)
    s = oracle.fold(rows)
    m = oracle.scale(s, oracle.mean_scale(W))
    r = M.recip(W)
    for i in range(400):
        assert int(as_bits(m)[i]) == M.mul(int(as_bits(s)[i]), r), i


@pytest.mark.parametrize("W", [2, 4, 8])
def test_power_of_two_mean_is_exact_quotient(W):
    rows = gen.gradient_rows(W, 1 << 14)
    s = oracle.fold(rows)
    m = oracle.scale(s, oracle.mean_scale(W))
    # normal-range sums: s / W is exact in binary64 and representable in binary32
    ok = np.abs(s) > 1e-30
    assert np.array_equal((s[ok].astype(np.float64) / W), m[ok].astype(np.float64))


def test_scale_one_is_identity():
    x = gen.stress_rows(1, 1000)[0]
    assert oracle.bit_diffs(oracle.scale(x, 1.0), x) == 0


# ---------------------------------------------------------------- shard plan

def _plan_by_dealing(length, W):
    # Independent construction: deal elements one at a time to owners in
    # round-robin, take the counts, and lay the shards out in rank order.
    counts = [0] * W
    for k in range(length):
        counts[k % W] += 1
    starts, s = [], 0
    for c in counts:
        starts.append(s)
        s += c
    return starts, counts


def test_shard_plan_brute_force():
    for W in range(1, 10):
        for length in range(0, 65):
            starts, lens = oracle.shard_plan(length, W)
            assert len(starts) == W
            assert starts[0] == 0 and int(lens.sum()) == length
            for r in range(W - 1):
                assert starts[r + 1] == starts[r] + lens[r]
            assert lens.max() - lens.min() <= 1
            ws, wl = _plan_by_dealing(length, W)
            assert list(starts) == ws and list(lens) == wl


def test_shard_plan_large():
    starts, lens = oracle.shard_plan(100_000_000, 4)
    assert list(lens) == [25_000_000] * 4
    assert list(starts) == [0, 25_000_000, 50_000_000, 75_000_000]
    starts, lens = oracle.shard_plan((1 << 20) + 7, 6)
    assert int(lens.sum()) == (1 << 20) + 7 and lens.max() - lens.min() == 1


# ---------------------------------------------------------------- all-reduce

@pytest.mark.parametrize("W,n", [(2, 33), (3, 50), (4, 64), (6, 41)])
def test_allreduce_end_state_matches_model(W, n):
    rows = gen.stress_rows(W, n)
    arenas = [rows[r].copy() for r in range(W)]
    scale = oracle.mean_scale(W)
    oracle.allreduce(arenas, scale)
    s = as_bits(model_fold(rows))
    want = np.array([M.mul(int(v), M.recip(W)) for v in s], dtype=np.uint32)
    for a in arenas:
        assert np.array_equal(as_bits(a), want)


@pytest.mark.parametrize("W", [1, 2, 3, 4, 6, 8])
@pytest.mark.parametrize("n", [0, 1, 2, 5, 7, 100, 4099])
@pytest.mark.parametrize("mean", [False, True])
def test_staged_dataflow_equals_fused(W, n, mean):
    rows = gen.stress_rows(W, n) if n else np.zeros((W, 0), np.float32)
    s = oracle.mean_scale(W) if mean else np.float32(1.0)
    fused = [rows[r].copy() for r in range(W)]
    oracle.allreduce(fused, s)
    for reverse in (False, True):
        staged = [rows[r].copy() for r in range(W)]
        oracle.staged_allreduce(staged, s, reverse=reverse)
        for r in range(W):
            assert oracle.bit_diffs(staged[r], fused[r]) == 0


def test_allreduce_repeat_call():
    # W = 2: after one call both arenas hold S, the second gives 2S exactly.
    n = 4096
    rows = gen.c1_rows(2, n)
    arenas = [rows[0].copy(), rows[1].copy()]
    oracle.allreduce(arenas)
    S = arenas[0].copy()
    oracle.allreduce(arenas)
    assert np.array_equal(arenas[0].astype(np.float64), 2.0 * S.astype(np.float64))


def test_bit_diffs_counts_exactly_the_differing_words():
    # the bench's checks count words with bit_diffs: it must compare bits, not
    # values (+0 vs -0 and two NaN payloads differ), and count each word once
    a = np.arange(1, 1001, dtype=np.float32)
    b = a.copy()
    assert oracle.bit_diffs(a, b) == 0
    b[[0, 17, 999]] = [np.float32(2.0), np.float32(-18.0), np.nextafter(np.float32(1000), np.float32(0))]
    assert oracle.bit_diffs(a, b) == 3
    z = np.zeros(4, dtype=np.float32)
    nz = z.copy()
    nz[2] = np.float32(-0.0)
    assert oracle.bit_diffs(z, nz) == 1
    n1 = np.array([0x7FC00001, 0x7FC00002], dtype=np.uint32).view(np.float32)
    assert oracle.bit_diffs(n1, n1.copy()) == 0
    assert oracle.bit_diffs(n1, n1[::-1].copy()) == 2
