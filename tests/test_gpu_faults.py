"""Failure detection on the GPU without a fault: a test hook makes CTA 0
skip the loads of its first pipeline stage, so the waits that depend on it
run out after a short, bounded timeout.  The kernel must come back (no
hang), report NVFP4_ERR_TIMEOUT through nvfp4_last_device_error, leave the
context usable, and the next call must be correct."""
import pytest

from gpu_util import compare_fp16, gemm_env, require_gb300
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", [None, "swap", "pair", "wide_sk"])
def test_expired_wait_reports_timeout_and_context_survives(kind):
    require_gb300()
    with gemm_env(kind):
        _expired_wait(kind)


def _expired_wait(kind):
    from block_scaled_nvfp4_group_gb300 import _abi, ops, workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    groups = workloads.make_groups([(200, 512, 2048), (64, 256, 1024)], seed=41)
    prob = DeviceProblem(groups)
    prob.relayout()
    assert ops.last_device_error() == _abi.NVFP4_OK
    ops.set_wait_timeout_ns(50_000_000)          # 50 ms per wait
    try:
        ops.debug_drop_first_stage(True)
        try:
            prob.gemm()
        finally:
            ops.debug_drop_first_stage(False)
        assert ops.last_device_error() == _abi.NVFP4_ERR_TIMEOUT
        assert ops.last_device_error() == _abi.NVFP4_OK      # read-and-clear
    finally:
        ops.set_wait_timeout_ns(2_000_000_000)
    for c in prob.C:
        c.fill_(float("nan"))
    prob.gemm()
    assert ops.last_device_error() == _abi.NVFP4_OK
    got = prob.outputs_fp16_bits()
    for g, c in zip(groups, got):
        compare_fp16(c, oracle.get().gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K), "after timeout")
