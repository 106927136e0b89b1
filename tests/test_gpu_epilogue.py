"""Fused epilogue of the grouped GEMM (per-group scale, BF16 output, SwiGLU
of 128-row gate / up blocks) against the oracle's epilogue of the exact
sums: FP16 within 1e-3 |C| + 1e-2, BF16 within 2^-7 |C| + 1e-2 (one BF16
ulp: the FP32 sum may round to the neighbour of the exact sum's BF16)."""
import numpy as np
import pytest
import torch

from gpu_util import compare_bf16, compare_fp16, gemm_env, require_gb300
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gb300()


def _run(groups, alpha, out_bf16, swiglu, kind=None):
    from block_scaled_nvfp4_group_gb300 import ops
    items = []
    for g in groups:
        A = torch.from_numpy(g.A).cuda().reshape(-1)
        B = torch.from_numpy(g.B).cuda().reshape(-1)
        sa = ops.sf_relayout(torch.from_numpy(g.SFA).cuda().reshape(-1), g.M, g.K)
        sb = ops.sf_relayout(torch.from_numpy(g.SFB).cuda().reshape(-1), g.N, g.K)
        n_out = g.N // 2 if swiglu else g.N
        C = torch.full((g.M, n_out), float("nan"), dtype=torch.bfloat16 if out_bf16 else torch.float16,
                       device="cuda")
        items.append((A, B, sa, sb, C, g.M, g.N, g.K))
    with gemm_env(kind):
        ops.group_gemm_ex(items, alpha=alpha, out_bf16=out_bf16, swiglu=swiglu)
    torch.cuda.synchronize()
    assert ops.last_device_error() == 0
    return [it[4].view(torch.int16).cpu().numpy().view(np.uint16) for it in items]


def _check(groups, alpha, out_bf16, swiglu, kind=None):
    o = oracle.get()
    got = _run(groups, alpha, out_bf16, swiglu, kind)
    for i, (g, c) in enumerate(zip(groups, got)):
        a = 1.0 if alpha is None else alpha[i]
        ref = o.gemm_ex(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, alpha=float(np.float32(a)),
                        swiglu=swiglu, bf16=out_bf16)
        what = f"group {i} {g.M}x{g.N}x{g.K} alpha={a} bf16={out_bf16} swiglu={swiglu} kind={kind}"
        (compare_bf16 if out_bf16 else compare_fp16)(c, ref, what)


SHAPES = [(200, 512, 1024), (77, 256, 512), (300, 768, 256), (1, 256, 2304)]


@pytest.mark.parametrize("kind", [None, "stream", "wide", "pair", "swap"])
def test_alpha_fp16(kind):
    from block_scaled_nvfp4_group_gb300 import workloads
    groups = workloads.make_groups(SHAPES, seed=51)
    _check(groups, [0.5, 0.0078125, 3.0, -1.25], False, False, kind)


@pytest.mark.parametrize("kind", [None, "pair", "swap"])
def test_bf16_output(kind):
    from block_scaled_nvfp4_group_gb300 import workloads
    groups = workloads.make_groups(SHAPES, seed=52)
    _check(groups, None, True, False, kind)
    _check(groups, [0.1, 0.2, 0.3, 0.4], True, False, kind)


@pytest.mark.parametrize("kind", [None, "wide", "pair", "stream", "swap"])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_swiglu(kind, out_bf16):
    """SwiGLU with small per-group scales (the gate/up sums of these inputs
    reach the hundreds; the products would overflow FP16 unscaled).  A
    forced 128-wide or swapped configuration falls back to the 256-wide
    one."""
    from block_scaled_nvfp4_group_gb300 import workloads
    groups = workloads.make_groups(SHAPES, seed=53)
    _check(groups, [1 / 64, 1 / 32, 1 / 128, 1 / 16], out_bf16, True, kind)


def test_moe_gate_up_swiglu_bf16():
    """The gate/up workload (K = 7168) through SwiGLU into BF16 on sampled
    rows of every group."""
    from block_scaled_nvfp4_group_gb300 import workloads
    o = oracle.get()
    wl = workloads.make_workload("moe_gate_up")
    alpha = [1 / 256] * len(wl.groups)
    got = _run(wl.groups, alpha, True, True)
    rng = np.random.default_rng(5)
    for i, (g, c) in enumerate(zip(wl.groups, got)):
        rows = sorted(set([0, g.M - 1] + rng.integers(0, g.M, size=6).tolist()))
        A = g.A[rows]
        SFA = g.SFA[rows]
        ref = o.gemm_ex(A, SFA, g.B, g.SFB, len(rows), g.N, g.K, alpha=alpha[i], swiglu=True, bf16=True)
        compare_bf16(c[rows], ref, f"moe_gate_up group {i} rows {rows}")


def test_plain_ex_matches_group_gemm():
    """With no options the extended entry point writes what nvfp4_group_gemm
    writes, bit for bit."""
    from block_scaled_nvfp4_group_gb300 import ops, workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    groups = workloads.make_groups(SHAPES, seed=54)
    prob = DeviceProblem(groups)
    prob.step()
    first = [c.clone() for c in prob.C]
    for c in prob.C:
        c.fill_(float("nan"))
    ops.group_gemm_ex(None, descs=prob.descs)
    torch.cuda.synchronize()
    for a, b in zip(first, prob.C):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_swiglu_rejects_ragged_n():
    from block_scaled_nvfp4_group_gb300 import _abi, ops, workloads
    groups = workloads.make_groups([(64, 384, 256)], seed=55)
    with pytest.raises(_abi.Nvfp4Error):
        _run(groups, None, False, True)


@pytest.mark.parametrize("kind", [None, "pair"])
def test_relayout_and_gemm_fused(kind):
    """The one-call path (nvfp4_relayout_and_gemm) from row-major scales, with
    per-group scales, BF16 output and SwiGLU, against the oracle."""
    from block_scaled_nvfp4_group_gb300 import ops, workloads
    groups = workloads.make_groups(SHAPES, seed=54)
    alpha = [1 / 64, 1 / 32, 1 / 128, 1 / 16]
    steps = []
    for g in groups:
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().reshape(-1)
        C = torch.full((g.M, g.N // 2), float("nan"), dtype=torch.bfloat16, device="cuda")
        steps.append((dev(g.A), dev(g.B), dev(g.SFA), dev(g.SFB),
                      torch.zeros(max(ops.sf_tiled_bytes(g.M, g.K), 16), dtype=torch.uint8, device="cuda"),
                      torch.zeros(max(ops.sf_tiled_bytes(g.N, g.K), 16), dtype=torch.uint8, device="cuda"),
                      C, g.M, g.N, g.K))
    with gemm_env(kind):
        ops.relayout_and_gemm(steps, alpha=alpha, out_bf16=True, swiglu=True)
    torch.cuda.synchronize()
    assert ops.last_device_error() == 0
    o = oracle.get()
    for i, (g, st) in enumerate(zip(groups, steps)):
        got = st[6].view(torch.int16).cpu().numpy().view(np.uint16)
        ref = o.gemm_ex(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, alpha=float(np.float32(alpha[i])),
                        swiglu=True, bf16=True)
        compare_bf16(got, ref, f"relayout+gemm group {i} kind={kind}")


def test_relayout_and_gemm_rejects_before_launch():
    """A missing row-major scale pointer is rejected before anything runs."""
    from block_scaled_nvfp4_group_gb300 import _abi
    lib = _abi.load()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    arr = (_abi.StepDesc * 1)()
    arr[0] = _abi.StepDesc(p, p, None, p, p, p, p, 128, 256, 256)
    assert lib.nvfp4_relayout_and_gemm(arr, 1, None, None) == _abi.NVFP4_ERR_INVALID_ARGUMENT
    arr[0] = _abi.StepDesc(p, p, p + 4, p, p, p, p, 128, 256, 256)
    assert lib.nvfp4_relayout_and_gemm(arr, 1, None, None) == _abi.NVFP4_ERR_MISALIGNED
