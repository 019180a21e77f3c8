"""bench.py's reference arm on the CPU: `--impl reference` times the oracle on the host cores and prints
one JSON line in the bench's format (metric, unit, steps, the cpu_baseline record and an e2e block
with no host-device traffic); ranks other than 0 print nothing."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ, **(extra_env or {}))
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny", "--steps", "2",
           "--warmup", "1", "--cpu-seconds", "0.5"]
    return subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)


def test_reference_arm_prints_one_line_in_the_bench_format():
    r = _run()
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["metric"].startswith("causal FP8 prefill attention TFLOP/s")
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"] and "rows" in cpu["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "B=1 H=2 H_kv=2 S=256" in d["config"]["workload"]


def test_reference_arm_other_ranks_do_no_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_e2e_record_names_the_library_chunk_plan():
    # the host-buffer entry point's plan for chunks = 0 (include/zyfa.h): from 32 query blocks of 256
    # rows, four equal chunks and two short tails; below that four equal chunks, at most one per block
    import bench
    assert bench.library_host_chunks(32768) == 6
    assert bench.library_host_chunks(32 * 256) == 6
    assert bench.library_host_chunks(31 * 256) == 4
    assert bench.library_host_chunks(4096) == 4
    assert bench.library_host_chunks(600) == 3
    assert bench.library_host_chunks(1) == 1
