"""Stream-K form of the 128 x 256 GEMM (kind WIDE_SK): every CTA takes an
equal contiguous range of the call's (tile, 256-K stage) units, so tiles are
cut between CTAs and the CTA holding a tile's first stages adds the others'
FP32 partial sums.  Checked against the oracle element by element (the
partial sums change the FP32 summation order only: same tolerance), for
tiles cut into two and into many pieces, ranges spanning whole tiles,
groups of different K, ragged M, the fused epilogue options, repeated calls
and CUDA-graph replays (the per-launch flag epoch)."""
import numpy as np
import pytest
import torch

from gpu_util import compare_fp16, gemm_env, require_gb300
from oracle import oracle
from test_gpu_epilogue import _check as check_epilogue
from test_gpu_gemm import run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gb300()


SPLITS = {
    # 64 tiles x 2 stages = 128 units on 128 CTAs: every tile in two pieces
    "two_pieces": [(1024, 2048, 512)],
    # 256 tiles x 2 stages on 152 CTAs: ranges of 3-4 units, whole tiles
    # inside ranges and tiles cut at both ends
    "mixed": [(2048, 4096, 512)],
    # 8 tiles x 28 stages on 152 CTAs: about 19 pieces per tile
    "many_helpers": [(256, 1024, 7168)],
    # groups of different K (stages per tile 1, 2, 4, 9), ragged M, an
    # empty group
    "ragged": [(200, 512, 1024), (77, 256, 256), (0, 256, 512), (300, 768, 512), (129, 256, 2304)],
    # the quantized workload's shape class: 96 tiles x 16 stages
    "quantized_like": [(512, 3072, 4096), (512, 3072, 4096)],
}


@pytest.mark.parametrize("name", list(SPLITS))
def test_stream_k_matches_oracle(name):
    from block_scaled_nvfp4_group_gb300 import workloads
    groups = workloads.make_groups(SPLITS[name], seed=71 + len(name))
    with gemm_env("wide_sk"):
        rows = 48 if name in ("mixed", "quantized_like") else None
        run_and_compare(groups, rows_per_group=rows, seed=7)


def test_stream_k_repeat_calls_identical():
    """The epoch moves on every launch; five calls give the same bits."""
    from block_scaled_nvfp4_group_gb300 import workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    groups = workloads.make_groups([(300, 768, 2048), (64, 512, 1024)], seed=72)
    prob = DeviceProblem(groups)
    prob.relayout()
    outs = []
    with gemm_env("wide_sk"):
        for _ in range(5):
            for c in prob.C:
                c.fill_(float("nan"))
            prob.gemm()
            torch.cuda.synchronize()
            outs.append(prob.outputs_fp16_bits())
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b)
    o = oracle.get()
    for g, c in zip(groups, outs[0]):
        compare_fp16(c, o.gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K), "stream-K repeat")


def test_stream_k_graph_replays_new_inputs():
    """A captured stream-K GEMM replayed with new operand bytes each time:
    the flags of one replay must never satisfy the next (the epoch lives in
    device memory, not in the captured parameters)."""
    from block_scaled_nvfp4_group_gb300 import workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    shapes = [(256, 1024, 4096), (130, 512, 1024)]
    prob = DeviceProblem(workloads.make_groups(shapes, seed=73))
    # the scratch of a stream is allocated by its first stream-K call, which
    # must not happen during capture: warm up on the capture stream
    cap = torch.cuda.Stream()
    with gemm_env("wide_sk"):
        prob.relayout()
        torch.cuda.synchronize()
        with torch.cuda.stream(cap):
            prob.gemm()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            prob.gemm()
    o = oracle.get()
    for rep in range(3):
        groups = workloads.make_groups(shapes, seed=100 + rep)
        for i, gr in enumerate(groups):
            prob.A[i].copy_(torch.from_numpy(np.ascontiguousarray(gr.A).reshape(-1)))
            prob.B[i].copy_(torch.from_numpy(np.ascontiguousarray(gr.B).reshape(-1)))
            prob.SFA[i].copy_(torch.from_numpy(np.ascontiguousarray(gr.SFA).reshape(-1)))
            prob.SFB[i].copy_(torch.from_numpy(np.ascontiguousarray(gr.SFB).reshape(-1)))
        prob.relayout()
        for c in prob.C:
            c.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for gr, c in zip(groups, prob.outputs_fp16_bits()):
            compare_fp16(c, o.gemm(gr.A, gr.SFA, gr.B, gr.SFB, gr.M, gr.N, gr.K), f"replay {rep}")


@pytest.mark.parametrize("out_bf16", [False, True])
def test_stream_k_fused_epilogue(out_bf16):
    """alpha and SwiGLU act on the whole sum: partials are added first."""
    from block_scaled_nvfp4_group_gb300 import workloads
    shapes = [(200, 512, 4096), (77, 256, 2048), (300, 768, 1024)]
    groups = workloads.make_groups(shapes, seed=74)
    check_epilogue(groups, [0.5, 3.0, -1.25], out_bf16, False, "wide_sk")
    check_epilogue(groups, [1 / 64, 1 / 32, 1 / 128], out_bf16, True, "wide_sk")


def test_plan_never_picks_stream_k_by_itself():
    """Stream-K runs only when forced (it measured slower than whole tiles on
    GB300, also for fewer tiles than SMs); forced, the plan reports it."""
    from block_scaled_nvfp4_group_gb300 import ops, workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem

    def plan(name):
        return ops.group_gemm_plan(descs=DeviceProblem(workloads.make_workload(name).groups).descs)

    for name in ("quantized", "moe_gate_up", "moe_down", "tiny"):
        assert plan(name)[0] != "wide_sk", name
    with gemm_env("wide_sk"):
        assert plan("quantized") == ("wide_sk", 1)
