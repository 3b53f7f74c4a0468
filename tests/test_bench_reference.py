"""bench.py on the CPU: the --impl reference arm (the oracle timed on the host cores) prints
one JSON line of the benchmark contract with the same config as the GPU arm, and a request
for more than one GPU is answered with one "unavailable" line (the library is single-GPU)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _run(*args):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_prints_one_contract_line():
    d = _run("--impl", "reference", "--workload", "prefill", "--steps", "1", "--warmup", "3")
    assert d["impl"] == "reference" and d["unit"] == "tok/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    import bench
    assert d["config"] == bench.config_of("prefill", 1)
    assert d["metric"] == bench.METRICS["prefill"]


def test_more_than_one_gpu_is_refused_with_one_line():
    d = _run("--gpus", "2", "--steps", "1", "--warmup", "3")
    assert d["n_gpus"] == 2 and "single-GPU" in d["unavailable"]


def test_headline_config_names_the_timed_cache_range():
    import bench
    c = bench.config_of("decode_bs1", 20)
    assert c["cache_start"] == 512 and c["cache_end"] == 532 and "512..531" in c["workload"]
    assert bench.config_of("decode_bs1", 256)["cache_end"] == 768
