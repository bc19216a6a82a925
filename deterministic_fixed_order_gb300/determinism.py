"""Determinism-diff harness for any libdetfold call.

After the determinism arm of memra-engine 0.123.0 src/bin/moe_tp2_repro.rs:
run the same call K times on identical inputs, count the output words that
differ from the first run, and refuse to call an all-zero result
deterministic. Zero data makes every accumulation order agree (the page's
RANDBANK note), so such a result is VACUOUS, not a pass.

Usage::

    report = determinism_diff(run=lambda k: df.detfold_sum_ptrs(out, srcs, W, n),
                              read=lambda k: out, repeats=8)
    assert report["verdict"] == "DETERMINISTIC"

Each callable receives the run index k. `reset(k)` restores identical inputs
before run k (needed for in-place calls such as the all-reduce), `run(k)`
enqueues the call, `read(k)` returns the output tensor (or a list of them).
Tensors may live on the CPU or a CUDA device; comparison is bitwise (int32
views), so NaN payloads and signed zeros count. With `streams`, run k goes
to streams[k % len(streams)] and all runs are enqueued before any is read,
so runs on different streams may overlap: the concurrent variant of the
arm. Give each run its own buffers there (index them by k).
"""
from __future__ import annotations

import torch


def _as_list(x):
    return list(x) if isinstance(x, (list, tuple)) else [x]


def _bits(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.float32:
        raise TypeError("determinism_diff compares float32 outputs")
    return t.contiguous().view(torch.int32)


def determinism_diff(run, read, reset=None, repeats: int = 8, streams=None) -> dict:
    if repeats < 2:
        raise ValueError("need at least two runs to compare")
    outs_all = []
    for k in range(repeats):
        ctx = torch.cuda.stream(streams[k % len(streams)]) if streams else _null()
        with ctx:
            if reset is not None:
                reset(k)
            run(k)
            if not streams:
                outs_all.append([o.clone() for o in _as_list(read(k))])
    if streams:
        torch.cuda.synchronize()
        outs_all = [[o.clone() for o in _as_list(read(k))] for k in range(repeats)]
    first = outs_all[0]
    diffs = [0]
    for outs in outs_all[1:]:
        if len(outs) != len(first) or any(a.shape != b.shape for a, b in zip(outs, first)):
            raise ValueError("read() changed shape between runs")
        diffs.append(int(sum(int((_bits(a) != _bits(b)).sum()) for a, b in zip(outs, first))))
    words = sum(o.numel() for o in first)
    nonzero = sum(int((o != 0).sum()) for o in first)
    nan = sum(int(torch.isnan(o).sum()) for o in first)
    finite = [o[torch.isfinite(o)] for o in first]
    absmax = max((float(f.abs().max()) for f in finite if f.numel()), default=0.0)
    if nonzero == 0:
        verdict = "VACUOUS"
    elif max(diffs) == 0:
        verdict = "DETERMINISTIC"
    else:
        verdict = "NONDETERMINISTIC"
    return {"runs": repeats, "words": words, "diff_words_per_run": diffs,
            "max_diff_words": max(diffs), "nonzero": nonzero, "nan": nan, "absmax": absmax,
            "verdict": verdict}


class _null:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False
