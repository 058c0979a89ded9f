"""Host-side checks of the benchmark harness (CPU only): the byte counts the
roofline divides by, the reference arm's JSON line (it times the CPU oracle,
so it runs here end to end on a tiny sample), rank > 0 doing no work, and
the warm-up floor."""
import json
import os
import subprocess
import sys

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def run_bench(*args, env=None, timeout=300):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          env=e, capture_output=True, text=True, timeout=timeout)


def test_algorithmic_bytes_closed_form():
    # 8B qkv at M = 1: packed weights (N K / 2 codes + N K / 16 scales),
    # packed X, two tensor scales, FP32 Y
    n, k = 6144, 4096
    b = bench.algorithmic_bytes(1, n, k)
    assert b["weights"] == n * k // 2 + n * k // 16 == 14_155_776
    assert b["gemm"] == 14_155_776 + k // 2 + k // 16 + 8 + 4 * n == 14_182_664
    assert b["quant"] == 4 * k + k // 2 + k // 16 + 4
    # BF16 I/O halves the X read and the Y write
    b16 = bench.algorithmic_bytes(8, n, k, 2, 2)
    assert b16["gemm"] == b16["weights"] + 8 * (k // 2 + k // 16) + 8 + 2 * 8 * n
    assert b16["quant"] == 2 * 8 * k + 8 * (k // 2 + k // 16) + 4
    # the 36-layer decode step's weights: 3.907 GB
    tot = sum(bench.algorithmic_bytes(1, l.n, l.k)["weights"] for l in bench.synthetic.LINEARS_8B)
    assert tot * 36 == 3_906_994_176


def test_reference_arm_prints_the_contract_line():
    r = run_bench("--impl", "reference", "--steps", "2", "--warmup", "3",
                  "--ref-step-seconds", "0.05")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_nothing():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3",
                  env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_warmup_floor():
    r = run_bench("--impl", "reference", "--warmup", "2")
    assert r.returncode == 2 and "warmup" in r.stderr
