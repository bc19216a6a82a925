"""The pin battery for a fold implementation on the CPU.

``fold_pin_failures(fold)`` runs a candidate fold (a callable taking a
``float32[W, n]`` array and returning ``float32[n]``) through checks whose
expected values come from outside the candidate:

* the hand-derived golden cases in ``tests/golden/hand_cases.txt``;
* the exact rational IEEE binary32 model of ``tests/ieee_model.py`` on
  seeded columns of every workload recipe;
* closed forms (all-ones, signed zeros, small integers, x + (-x));
* the double-simulated chain on larger arrays: each partial sum computed in
  binary64 and rounded to binary32, which equals the binary32 chain because
  double rounding is innocuous for addition when the wider format has at
  least 2p + 2 significand bits (53 >= 2*24 + 2; S. A. Figueroa,
  "When is double rounding innocuous?", ACM SIGNUM Newsletter 30(3), 1995).

The same battery is run on planted mutants of the oracle (reversed order,
accumulator started at +0, a dropped rank, a wider accumulator, a pairwise
tree, flush-to-zero, a shifted index) to show that every such mistake fails
at least one pin.
"""
from __future__ import annotations

import os

import numpy as np

import detfold_inputs as gen
from ieee_model import chain

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_cases.txt")


def load_hand_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, W, addends, s, mean = line.split()
            adds = [int(h, 16) for h in addends.split(",")]
            assert len(adds) == int(W), name
            cases.append((name, int(W), adds, int(s, 16), None if mean == "-" else int(mean, 16)))
    return cases


def bits_array(bits: list[int]) -> np.ndarray:
    return np.array(bits, dtype=np.uint32).view(np.float32)


def as_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def _check_golden(fold, fails):
    for name, W, adds, want, _ in load_hand_cases():
        rows = bits_array(adds).reshape(W, 1)
        got = int(as_bits(fold(rows))[0])
        if got != want:
            fails.append(f"golden {name}: got {got:08x} want {want:08x}")


def model_fold(rows: np.ndarray) -> np.ndarray:
    """Exact-model ascending chain per column (slow: small inputs only)."""
    b = as_bits(rows)
    W, n = b.shape
    out = np.empty(n, dtype=np.uint32)
    for i in range(n):
        out[i] = chain([int(b[r, i]) for r in range(W)])
    return out.view(np.float32)


def _check_model(fold, fails, n=48):
    for recipe in ("vecf", "gradient", "normal", "stress"):
        for W in (2, 3, 4, 6, 8):
            rows = gen.recipe_rows(recipe, W, 4096)
            # the first columns carry the stress specials; add a strided sample
            idx = np.r_[0:16, np.linspace(16, 4095, n - 16).astype(np.int64)]
            sub = np.ascontiguousarray(rows[:, idx])
            want = as_bits(model_fold(sub))
            got = as_bits(fold(sub))
            bad = np.nonzero(got != want)[0]
            if bad.size:
                i = bad[0]
                fails.append(f"model {recipe} W={W}: {bad.size} columns differ, first col {idx[i]}"
                             f" got {got[i]:08x} want {want[i]:08x}")


def _check_closed_forms(fold, fails):
    for W in range(1, 65):
        got = fold(np.ones((W, 3), dtype=np.float32))
        if not np.all(got == np.float32(W)):
            fails.append(f"closed all-ones W={W}: got {got[0]!r}")
            break
    negz = np.full((5, 4), -0.0, dtype=np.float32)
    got = as_bits(fold(negz))
    if not np.all(got == 0x80000000):
        fails.append("closed all -0 column is not -0")
    rng = np.random.default_rng(7)
    ints = rng.integers(-2000, 2000, size=(8, 512)).astype(np.float32)
    want = ints.astype(np.int64).sum(axis=0).astype(np.float32)  # |partials| < 2^24: exact
    if not np.array_equal(as_bits(fold(ints)), as_bits(want)):
        fails.append("closed small-integer sums are not exact")
    x = gen.normal_rows(1, 256)[0]
    got = as_bits(fold(np.stack([x, -x])))
    if not np.all(got == 0):
        fails.append("closed x + (-x) is not +0 everywhere")


def double_simulated_fold(rows: np.ndarray) -> np.ndarray:
    """Each partial in binary64, rounded to binary32 after every add."""
    acc = rows[0].astype(np.float32)
    for r in range(1, rows.shape[0]):
        acc = (acc.astype(np.float64) + rows[r].astype(np.float64)).astype(np.float32)
    return acc


def _check_double_sim(fold, fails, n=1 << 16):
    for recipe, W in (("gradient", 8), ("stress", 6), ("stress", 3), ("normal", 4), ("vecf", 2)):
        rows = gen.recipe_rows(recipe, W, n)
        want = as_bits(double_simulated_fold(rows))
        got = as_bits(fold(rows))
        d = int(np.count_nonzero(got != want))
        if d:
            fails.append(f"double-sim {recipe} W={W}: {d} of {n} words differ")


def fold_pin_failures(fold) -> list[str]:
    fails: list[str] = []
    _check_golden(fold, fails)
    _check_closed_forms(fold, fails)
    _check_model(fold, fails)
    _check_double_sim(fold, fails)
    return fails


# ---------------------------------------------------------------------------
# Planted mutants of the oracle (CPU only): each is a plausible mistake.

def _mut_reverse(rows):
    return double_simulated_fold(np.ascontiguousarray(rows[::-1]))


def _mut_zero_start(rows):
    acc = np.zeros(rows.shape[1], dtype=np.float32)
    for r in range(rows.shape[0]):
        acc = acc + rows[r]
    return acc


def _mut_drop_last(rows):
    if rows.shape[0] == 1:
        return rows[0].copy()
    return double_simulated_fold(np.ascontiguousarray(rows[:-1]))


def _mut_wide_acc(rows):
    return rows.astype(np.float64).sum(axis=0).astype(np.float32)


def _mut_pairwise(rows):
    cur = [rows[r].astype(np.float32) for r in range(rows.shape[0])]
    while len(cur) > 1:
        nxt = [cur[k] + cur[k + 1] for k in range(0, len(cur) - 1, 2)]
        if len(cur) % 2:
            nxt.append(cur[-1])
        cur = nxt
    return cur[0]


def _mut_ftz(rows):
    acc = rows[0].astype(np.float32).copy()
    for r in range(1, rows.shape[0]):
        acc = acc + rows[r]
        tiny = np.abs(acc) < np.float32(1.1754944e-38)
        acc[tiny] = np.float32(0.0) * np.sign(acc[tiny])
    return acc


def _mut_shift(rows):
    out = double_simulated_fold(rows)
    if rows.shape[1] > 1:
        out = out.copy()
        out[1:] = double_simulated_fold(np.ascontiguousarray(np.concatenate(
            [rows[:1, 1:], rows[1:, :-1]], axis=0)))
    return out


def _mut_rank0_twice(rows):
    if rows.shape[0] < 2:
        return rows[0].copy()
    r = rows.copy()
    r[1] = r[0]
    return double_simulated_fold(r)


MUTANTS = {
    "reverse_order": _mut_reverse,
    "zero_start": _mut_zero_start,
    "drop_last_rank": _mut_drop_last,
    "wide_accumulator": _mut_wide_acc,
    "pairwise_tree": _mut_pairwise,
    "flush_to_zero": _mut_ftz,
    "shifted_index": _mut_shift,
    "rank0_twice": _mut_rank0_twice,
}
