"""bench.py's JSON contract on the CPU: the reference arm (the FP64 oracle,
timed on the host) prints one JSON line with the benchmark contract's keys, and the
argument checks reject combinations the library does not run."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=300):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT)


def test_reference_arm_line():
    r = _run("--impl", "reference", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["metric"].startswith("paged decode attention KV GB/s")
    assert d["config"]["workload"].startswith("ragged-b256")
    assert d["config"]["batch"] == 256 and d["config"]["layers"] == 16
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert cb["nproc"] >= cb["cores"] and cb["cpu_model"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == "GB/s"
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_rejects_options_the_multi_layer_launch_does_not_take():
    for extra in (("--rope",), ("--splits", "4")):
        r = _run("--persistent", *extra, "--steps", "1", "--warmup", "3")
        assert r.returncode != 0 and "--persistent" in r.stderr


def test_cpu_baseline_reports_single_thread_and_all_cores():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    cb = bench.cpu_baseline(W.custom([300, 17, 2048], num_layers=2, seed=7), seconds=0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["cpu_model"]
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert cb["all_cores"]["cores"] >= 1 and cb["nproc"] == (os.cpu_count() or 1)
    assert cb["value"] == cb["all_cores"]["value"] and cb["cores"] == cb["all_cores"]["cores"]


def test_oracle_sample_keeps_the_length_mix():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    wl = W.large_ragged()
    sw = bench.oracle_sample(wl)
    assert sw.batch == 64 and sw.num_layers == 4
    assert (sw.seq_lens == wl.seq_lens[:64]).all() and sw.k_scale == wl.k_scale
    assert bench.step_bytes(sw) // 4 == bench.step_bytes(W.custom(wl.seq_lens[:64]))


def test_algorithmic_bytes():
    """Per (sequence, layer): seq_len x 2048 (every K/V row read once, the new
    one included) + 2048 (the new row written) + 4096 (q) + 8192 (FP32 out),
    + 256 with rotary tables (two 32-float angle rows)."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    wl = W.llama_default()
    assert bench.step_bytes(wl) == 16 * 2 * (2048 * 2048 + 2048 + 4096 + 8192) == 134_676_480
    assert bench.step_bytes(wl, rope=True) == 134_676_480 + 16 * 2 * 256
    wl = W.custom([1, 17, 2048], num_layers=3)
    assert bench.step_bytes(wl) == 3 * sum(n * 2048 + 14336 for n in (1, 17, 2048))
