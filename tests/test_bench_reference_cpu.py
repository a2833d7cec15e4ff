"""bench.py's host-side logic without a GPU: the reference arm (the oracle
stepping whole layer-steps on the host cores) prints one JSON line with
every key the benchmark contract asks for, on the tiny workload; the
whole-step rates of the GPU arm's line are its bytes times its step rate."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line_has_the_contract_keys():
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(p.stdout.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert set(line["config"]) == {"workload", "parallelism", "l2"}
    assert line["config"]["workload"].startswith("tiny:")
    assert "smaller than L2" in line["config"]["l2"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    e = line["e2e"]
    assert e["value"] == line["value"] and e["unit"] == line["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_whole_step_rates():
    import bench
    pk = {"attention": {"bytes_per_step": 1_000_000}, "summary_scan": {"bytes_per_step": 500_000}}
    r = bench.whole_step_rates(pk, 50_000, 2000.0, {"hbm_gbs": 6.0}, 0.2)
    assert r["hbm_bytes_per_step"] == 1_500_000 and r["link_bytes_per_step"] == 50_000
    assert r["hbm_gbs"] == 3.0 and r["hbm_frac"] == 0.5        # 1.5 MB x 2000 / s
    assert r["link_gbs"] == 0.1 and r["link_frac"] == 0.5       # 50 kB x 2000 / s
