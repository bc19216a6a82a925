"""The determinism-diff harness's verdict logic, on the CPU (no GPU needed).

After the determinism arm of memra-engine 0.123.0 src/bin/moe_tp2_repro.rs:
identical runs must agree word for word, a differing run is reported with
its word count, and an all-zero result is VACUOUS rather than a pass.
"""
import importlib.util
import os

import pytest
import torch

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _harness():
    # loaded by path: the module needs only torch, not the built library
    spec = importlib.util.spec_from_file_location(
        "_det", os.path.join(_ROOT, "deterministic_fixed_order_gb300", "determinism.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m.determinism_diff


def test_identical_runs_are_deterministic():
    dd = _harness()
    x = torch.linspace(-3, 5, 1000)
    out = torch.empty(1000)
    r = dd(run=lambda k: torch.mul(x, 3.0, out=out), read=lambda k: out, repeats=5)
    assert r["verdict"] == "DETERMINISTIC" and r["max_diff_words"] == 0
    assert r["nonzero"] > 0 and r["absmax"] == 15.0


def test_order_dependent_runs_are_caught():
    dd = _harness()
    rows = torch.tensor([[1.0e8] * 64, [1.0] * 64, [-1.0e8] * 64], dtype=torch.float32)
    out = torch.empty(64)

    def run(k):
        order = [0, 2, 1] if k % 2 == 0 else [0, 1, 2]   # a different rank order on odd runs
        acc = rows[order[0]].clone()
        for r in order[1:]:
            acc = acc + rows[r]
        out.copy_(acc)

    r = dd(run=run, read=lambda k: out, repeats=4)
    assert r["verdict"] == "NONDETERMINISTIC"
    assert r["diff_words_per_run"] == [0, 64, 0, 64]


def test_all_zero_output_is_vacuous():
    dd = _harness()
    out = torch.zeros(100)
    r = dd(run=lambda k: out.zero_(), read=lambda k: out, repeats=3)
    assert r["verdict"] == "VACUOUS"


def test_signed_zero_and_nan_payloads_count_as_differences():
    dd = _harness()
    out = torch.ones(4)

    def run(k):
        out.view(torch.int32)[0] = 0x7FC00001 + k   # NaN with a run-dependent payload
    r = dd(run=run, read=lambda k: out, repeats=3)
    assert r["verdict"] == "NONDETERMINISTIC" and r["nan"] == 1


def test_needs_two_runs():
    dd = _harness()
    with pytest.raises(ValueError):
        dd(run=lambda k: None, read=lambda k: torch.ones(1), repeats=1)
