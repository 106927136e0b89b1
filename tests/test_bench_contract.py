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


def test_rotating_copies_exceed_twice_the_l2():
    """Between two uses of one copy's inputs the other copies' inputs total
    at least 2 x L2; workloads needing more than 64 copies flush instead."""
    sys.path.insert(0, ROOT)
    import bench
    for nbytes in (69 * 10**6, 140 * 10**6, 15 * 10**6, 300 * 10**6):
        r = bench.copies_needed(nbytes)
        assert r >= 2 and (r - 1) * nbytes >= 2 * bench.L2_BYTES
        assert (r - 2) * nbytes < 2 * bench.L2_BYTES        # no more copies than needed
    assert bench.copies_needed(200 * 10**3) == 0             # tiny: flush protocol


def test_roofline_and_summary_arithmetic():
    """The roofline picks the larger of the byte and FLOP times, divides the
    algorithmic work per launch by the mean launch time, and the summary's
    value is FLOPs per step time."""
    sys.path.insert(0, ROOT)
    import bench
    from block_scaled_nvfp4_group_gb300 import workloads
    peaks = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0, "source": "test"}

    def rec(name, shapes, gemm_ms, launches=1):
        return {"name": name, "flops": bench.flops_of(shapes), "gemm_bytes": bench.bytes_of(shapes),
                "gemm_ms": gemm_ms * launches, "launches_per_step": 1 + launches, "kernel": "k", "kind": "wide"}

    moe = workloads.describe("moe_gate_up")["shapes"]
    r = bench.roofline_of(rec("moe_gate_up", moe, 0.05), peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - bench.bytes_of(moe) / 50e-6 / 1e9) < 1e-6 * r["achieved"]
    assert abs(r["frac"] - r["achieved"] / 8000.0) < 1e-12
    sq = workloads.describe("square")["shapes"]
    r = bench.roofline_of(rec("square", sq, 0.1), peaks)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0 * 6
    assert abs(r["achieved"] - bench.flops_of(sq) / 100e-6 / 1e12) < 1e-6 * r["achieved"]
    # two GEMM launches per call: the per-launch time halves the call's
    r2 = bench.roofline_of(rec("square", sq, 0.1, launches=2), peaks)
    assert abs(r2["launch_us"] - 100.0) < 1e-9
    # traffic only while the recorded counters describe these sources
    assert (r["traffic"] is not None) == (bench.NCU_TRAFFIC["square"]["kernel_sha"] == bench.kernel_source_hash())
    assert bench.bytes_of([(0, 256, 256)]) == 0
