"""Host-side pieces of bench.py, checked without a GPU: the byte accounting
of every row, the peak lookup, the kernel-source hash and the reference arm."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_row_bytes_follow_the_algorithmic_formulas():
    b = bench.row_bytes()
    assert b["c3_stacked"] == 9 * (1 << 26) * 4 == 2_415_919_104
    assert b["c4_fused"] == b["c4_staged"] == 2 * 4 * 100_000_000 * 4
    n5 = (1 << 20) + 7
    assert b["c5_w3"] == (4 + 2 + 6) * n5 * 4
    assert b["c5_w6"] == (7 + 2 + 12) * n5 * 4
    assert b["c2_4096"] == 3 * 4096 * 4


def test_step_input_bytes_count_each_input_once():
    # the end-to-end leg uploads exactly these bytes per step (asserted in
    # bench.py): C3 8 x 2^26, C4 4 x 1e8, C5 (3 + 6) x (2^20 + 7), C2 2 x n
    n5 = (1 << 20) + 7
    want = 4 * (8 * (1 << 26) + 4 * 100_000_000 + 9 * n5 + 2 * (4096 + 65536))
    assert bench.step_input_bytes() == want == 3_785_789_692


def test_kernel_hash_covers_existing_files_and_is_stable():
    h1, h2 = bench.kernel_source_hash(), bench.kernel_source_hash()
    assert h1 == h2 and len(h1) == 16
    for f in bench.KERNEL_FILES:
        assert os.path.exists(os.path.join(ROOT, "deterministic_fixed_order_gb300", "csrc", f))


def test_peak_lookup_has_a_named_source():
    peak, src = bench.peaks()
    assert peak > 1000 and src in ("measured", "fallback")


def test_whole_job_value():
    assert abs(bench.whole_job_gbs(2, 10_000_000_000, 2.0) - 10_000.0) < 1e-9


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_verify_samples_counts_differing_words():
    # the oracle leg's check of collected samples: exact outputs give 0, and a
    # planted wrong word is counted once per sample it sits in
    import numpy as np

    import detfold_inputs as gen
    import oracle
    rows = gen.stress_rows(3, 257)
    fold = oracle.fold(rows)
    scale = oracle.mean_scale(3)
    arenas = [r.copy() for r in rows]
    for _ in range(2):
        oracle.allreduce(arenas, scale)
    specs = [
        {"group": "a", "kind": "fold_stacked", "inputs": rows, "got": [fold.copy(), fold.copy()]},
        {"group": "b", "kind": "fold_scale", "inputs": rows, "scale": scale,
         "got": [oracle.scale(fold, scale)]},
        {"group": "c", "kind": "allreduce", "repeat": 2, "scale": scale,
         "inputs": [r.copy() for r in rows], "got": [[a.copy() for a in arenas]]},
    ]
    assert bench.verify_samples(oracle, specs) == {"a": 0, "b": 0, "c": 0}
    specs[0]["got"][1][5] = np.nextafter(specs[0]["got"][1][5], np.float32(np.inf))
    specs[2]["got"][0][2][100] = -specs[2]["got"][0][2][100] if specs[2]["got"][0][2][100] != 0 else 1.0
    assert bench.verify_samples(oracle, specs) == {"a": 1, "b": 0, "c": 1}
    # the inputs are left as they were (the repeated all-reduce works on copies)
    assert all(np.array_equal(a.view(np.uint32), r.view(np.uint32)) for a, r in zip(specs[2]["inputs"], rows))


def test_gpu_arm_calls_the_oracle_only_through_its_oracle_leg():
    # bench.py may use the CPU oracle only to time it and to check samples:
    # run_gpu itself holds no oracle call
    import ast
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    fn = next(n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name == "run_gpu")
    names = {n.id for n in ast.walk(fn) if isinstance(n, ast.Name)}
    attrs = {n.value.id for n in ast.walk(fn)
             if isinstance(n, ast.Attribute) and isinstance(n.value, ast.Name)}
    imports = {a.name for n in ast.walk(fn) if isinstance(n, (ast.Import, ast.ImportFrom))
               for a in n.names}
    assert "oracle" not in names | attrs | imports
