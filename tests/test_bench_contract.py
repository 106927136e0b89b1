"""bench.py on a machine without a GPU: the reference arm (the CPU oracle)
prints one JSON line with the contract's keys, and the GPU arm fails loudly
instead of falling back to the CPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=300):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_one_contract_line():
    r = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # the same metric, unit and config as the GPU arm's line for this workload
    assert d["unit"] == "TFLOPS"
    assert d["config"]["M_g"] == [64, 128] and d["config"]["N"] == 256 and d["config"]["K"] == 256


def test_gpu_arm_fails_without_a_gpu():
    r = _run("--workload", "tiny", "--steps", "1", "--warmup", "3")
    assert r.returncode != 0
    assert not any(ln.lstrip().startswith("{") for ln in r.stdout.splitlines())


def test_oracle_sample_and_parity_count():
    """The CPU-baseline leg keeps the oracle rows it timed, and the bench's
    mismatch count flags a planted error (CPU only: both sides here are the
    oracle)."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from block_scaled_nvfp4_group_gb300 import workloads
    wl = workloads.make_workload("tiny")
    rate, desc, cores, dt, kept = bench.time_oracle(wl, 0.05, keep=True)
    assert rate > 0 and cores >= 1
    assert [gi for gi, _, _ in kept] == [0, 1]
    for gi, rows, ref in kept:
        g = wl.groups[gi]
        assert ref.shape == (rows.size, g.N) and rows.min() >= 0 and rows.max() < g.M
        assert bench.fp16_mismatches(ref, ref) == 0
        worse = ref.copy()
        v = worse.view(np.float16)
        v[0, 0] = np.float16(float(v[0, 0]) + 1.0 + 0.01 * abs(float(v[0, 0])))
        assert bench.fp16_mismatches(worse, ref) == 1
    assert bench.time_oracle(wl, 0.05)[4] is None
