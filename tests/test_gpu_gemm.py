"""Grouped GEMM on the GPU against the CPU oracle, element by element,
within |C - C_oracle| <= 1e-3 |C_oracle| + 1e-2 (the FP32 tensor-core sum is
rounded once more than the exact float64 sum; one FP16 ulp is at most 2^-10
relative)."""
import numpy as np
import pytest
import torch

from gpu_util import compare_fp16, gemm_env, require_gb300
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gb300()


def run_and_compare(groups, rows_per_group=None, seed=0):
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    prob = DeviceProblem(groups)
    for c in prob.C:                   # garbage in C: every element must be written
        c.fill_(float("nan"))
    prob.step()
    torch.cuda.synchronize()
    got = prob.outputs_fp16_bits()
    o = oracle.get()
    rng = np.random.default_rng(seed)
    for i, (g, c) in enumerate(zip(groups, got)):
        if g.M == 0:
            continue
        if rows_per_group is None:
            ref = o.gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K)
            compare_fp16(c, ref, f"group {i} ({g.M}x{g.N}x{g.K})")
        else:
            rows = sorted(set([0, g.M - 1, min(127, g.M - 1), min(128, g.M - 1)] +
                              rng.integers(0, g.M, size=rows_per_group).tolist()))
            ref = o.gemm_rows(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, rows)
            compare_fp16(c[rows], ref, f"group {i} rows {len(rows)} ({g.M}x{g.N}x{g.K})")
    return prob


def test_small_single_tile():
    from block_scaled_nvfp4_group_gb300 import workloads
    run_and_compare(workloads.make_groups([(128, 128, 256)], seed=1))


@pytest.mark.parametrize("kind", ["stream", "compute"])
def test_ragged_several_tiles(kind):
    """Several M and N tiles per group, ragged tails in M and N, one-stage
    and multi-stage K (K % 512 == 256 too: a half last stage), an empty
    group in the middle."""
    from block_scaled_nvfp4_group_gb300 import workloads
    shapes = [(200, 384, 1024), (77, 256, 512), (0, 256, 256), (1, 136, 256), (300, 520, 768),
              (129, 8, 2048)]
    with gemm_env(kind):
        run_and_compare(workloads.make_groups(shapes, seed=2))


@pytest.mark.parametrize("kind", ["wide", "wide512", "wide_p2", "wide_p4"])
def test_wide_tiles_ragged_m(kind):
    """BN = 256 tiles (two scale blocks per B tile), ragged M, several N
    tiles, one- and multi-stage K, half last stages."""
    from block_scaled_nvfp4_group_gb300 import workloads
    shapes = [(77, 512, 1024), (300, 256, 512), (1, 768, 256), (129, 1024, 2304)]
    with gemm_env(kind):
        run_and_compare(workloads.make_groups(shapes, seed=21))


@pytest.mark.parametrize("kind,pf", [("stream", 0), ("stream", 8), ("stream", 40), ("wide", 0),
                                     ("wide", 8), ("wide512", 0), ("compute", 0), ("pair", 0),
                                     ("pair", 2), ("pair", 12)])
def test_more_stages_than_ring_and_many_tiles(kind, pf):
    """K large enough to wrap the shared-memory ring several times per tile
    and more tiles than SMs (persistent loop, both accumulator buffers), with
    the L2 prefetch of B off, on, and running across tile boundaries."""
    from block_scaled_nvfp4_group_gb300 import workloads
    shapes = [(384, 2048, 4096), (256, 4096, 2560)]
    with gemm_env(kind, pf):
        run_and_compare(workloads.make_groups(shapes, seed=3))


def test_pair_tiles_ragged():
    """CTA pairs (256 x 256 tiles): M tails that leave the odd CTA of a pair
    with no rows (M <= 128 past a 256 boundary), N not a multiple of 256 (the
    odd CTA's B half partly or wholly past N), an empty group, one- and
    multi-stage K, more tiles than pairs."""
    from block_scaled_nvfp4_group_gb300 import workloads
    shapes = [(200, 384, 1024), (77, 256, 512), (0, 256, 256), (1, 264, 256), (300, 520, 768),
              (513, 1024, 2304), (129, 2048, 256)]
    with gemm_env("pair"):
        run_and_compare(workloads.make_groups(shapes, seed=22))


@pytest.mark.parametrize("kind", [None, "swap"])
def test_more_groups_than_one_launch(kind):
    from block_scaled_nvfp4_group_gb300 import workloads
    rng = np.random.default_rng(4)
    shapes = [(int(rng.integers(1, 200)), 8 * int(rng.integers(1, 40)), 256 * int(rng.integers(1, 4)))
              for _ in range(40)]
    with gemm_env(kind):
        run_and_compare(workloads.make_groups(shapes, seed=4))


@pytest.mark.parametrize("pf", [None, 0, 2])
def test_swap_token_tiles_ragged(pf):
    """The transposed product on CTA pairs: token tiles of every size class
    (1, 5, 45 rows: MMA N = 16..48; 129: two token scale blocks; 256 and
    257: one full tile and a split into 128 + 129; 385, 513: tiles of 256
    and a remainder), N past the 256 grid (264, 520: the odd CTA's rows of B
    partly or wholly past N), N below 256, one- and multi-stage K, an empty
    group, more tiles than pairs; with the L2 prefetch of B off and on."""
    from block_scaled_nvfp4_group_gb300 import workloads
    shapes = [(1, 256, 256), (5, 512, 768), (45, 256, 2304), (77, 264, 512), (0, 256, 256),
              (129, 768, 256), (200, 256, 1024), (256, 512, 512), (257, 256, 256), (300, 520, 768),
              (385, 256, 512), (513, 256, 256), (64, 136, 256), (7, 8, 256)]
    with gemm_env("swap", pf):
        run_and_compare(workloads.make_groups(shapes, seed=23))


def test_swap_many_token_tiles_and_launches():
    """A forced swapped call whose groups need more token tiles than one
    launch holds (1100 rows = 5 token tiles each; 20 groups), so groups
    continue across launches, with K wrapping the ring several times."""
    from block_scaled_nvfp4_group_gb300 import workloads
    shapes = [(1100, 256, 1536)] * 7 + [(97, 512, 256)] * 13
    with gemm_env("swap"):
        run_and_compare(workloads.make_groups(shapes, seed=24), rows_per_group=40, seed=5)


def test_full_scale_range_and_signs():
    """Scales over every finite positive E4M3FN value, sign-carrying codes:
    magnitudes far from 1 and overflow to inf in FP16 on both sides."""
    from block_scaled_nvfp4_group_gb300.workloads import Group
    rng = np.random.default_rng(6)
    groups = []
    for (M, N, K) in [(130, 200, 512), (64, 64, 256)]:
        pool = np.array([b for b in range(1, 0x7F)], dtype=np.uint8)
        groups.append(Group(M, N, K,
                            rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8),
                            rng.choice(pool, size=(M, K // 16)),
                            rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8),
                            rng.choice(pool, size=(N, K // 16))))
    run_and_compare(groups)


def test_output_bounds_untouched():
    """The TMA store clips at M and N: bytes around each C stay intact."""
    from block_scaled_nvfp4_group_gb300 import ops, workloads
    groups = workloads.make_groups([(77, 136, 512), (5, 8, 256)], seed=7)
    items, guards = [], []
    for g in groups:
        A = torch.from_numpy(g.A).cuda().reshape(-1)
        B = torch.from_numpy(g.B).cuda().reshape(-1)
        sa = ops.sf_relayout(torch.from_numpy(g.SFA).cuda().reshape(-1), g.M, g.K)
        sb = ops.sf_relayout(torch.from_numpy(g.SFB).cuda().reshape(-1), g.N, g.K)
        pad = 4096
        buf = torch.full((pad + g.M * g.N + pad,), 1234.0, dtype=torch.float16, device="cuda")
        C = buf[pad:pad + g.M * g.N].view(g.M, g.N)
        items.append((A, B, sa, sb, C, g.M, g.N, g.K))
        guards.append((buf, pad))
    ops.group_gemm(items)
    torch.cuda.synchronize()
    o = oracle.get()
    for g, (buf, pad), it in zip(groups, guards, items):
        b = buf.cpu()
        assert (b[:pad] == 1234.0).all() and (b[pad + g.M * g.N:] == 1234.0).all()
        ref = o.gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K)
        compare_fp16(it[4].view(torch.int16).cpu().numpy().view(np.uint16), ref, "guarded")


def test_repeat_calls_identical():
    from block_scaled_nvfp4_group_gb300 import workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    prob = DeviceProblem(workloads.make_groups([(300, 1024, 2048)] * 3, seed=8))
    prob.step()
    first = [c.clone() for c in prob.C]
    for _ in range(3):
        prob.step()
    torch.cuda.synchronize()
    for a, b in zip(first, prob.C):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("kind", [None, "pair", "stream"])
def test_l2_hints_and_prefetch_leave_results_unchanged(kind, monkeypatch):
    """The L2 eviction hint for B (normal / evict-first / evict-last) and the
    optional L2 prefetch of B are performance settings only: every setting
    gives bit-identical C, equal to the oracle's within the tolerance."""
    from block_scaled_nvfp4_group_gb300 import workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    groups = workloads.make_groups([(64, 4096, 1024)] * 8 + [(190, 512, 2048)], seed=31)
    ref = None
    with gemm_env(kind):
        run_and_compare(groups, rows_per_group=8, seed=3)
        prob = DeviceProblem(groups)
        for policy, pf in [("0", "0"), ("1", "0"), ("2", "0"), ("2", "3")]:
            monkeypatch.setenv("NVFP4_B_POLICY", policy)
            monkeypatch.setenv("NVFP4_PF_STAGES", pf)
            for c in prob.C:
                c.fill_(float("nan"))
            prob.step()
            torch.cuda.synchronize()
            out = [c.clone().view(torch.int16) for c in prob.C]
            if ref is None:
                ref = out
            else:
                for a, b in zip(ref, out):
                    assert torch.equal(a, b), (policy, pf)


# --- the benchmark workloads, in the launch configuration bench.py times -----

def test_workload_tiny():
    from block_scaled_nvfp4_group_gb300 import workloads
    run_and_compare(workloads.make_workload("tiny").groups)


@pytest.mark.parametrize("kind", [None, "wide", "pair", "swap"])
def test_workload_quantized(kind):
    from block_scaled_nvfp4_group_gb300 import workloads
    with gemm_env(kind):
        run_and_compare(workloads.make_workload("quantized").groups)


@pytest.mark.parametrize("kind", [None, "swap", "stream", "wide512", "compute", "pair", "wide_sk"])
def test_workload_moe_down(kind):
    from block_scaled_nvfp4_group_gb300 import workloads
    with gemm_env(kind):
        run_and_compare(workloads.make_workload("moe_down").groups)


@pytest.mark.parametrize("kind", [None, "swap", "stream", "wide512", "compute", "pair"])
def test_workload_moe_gate_up(kind):
    from block_scaled_nvfp4_group_gb300 import workloads
    with gemm_env(kind):
        run_and_compare(workloads.make_workload("moe_gate_up").groups)


@pytest.mark.parametrize("kind", [None, "wide", "pair"])
def test_workload_square_sampled_rows(kind):
    from block_scaled_nvfp4_group_gb300 import workloads
    with gemm_env(kind):
        run_and_compare(workloads.make_workload("square").groups, rows_per_group=24, seed=9)


@pytest.mark.parametrize("kind", [None, "pair", "swap"])
def test_step_graph_replays_new_inputs(kind):
    """The step as bench.py times it: one nvfp4_relayout_and_gemm call (scale
    relayout + grouped GEMM) captured as a CUDA graph on a side stream and
    replayed, with new operand bytes and new row-major scales before every
    replay; C is poisoned before each one."""
    from block_scaled_nvfp4_group_gb300 import workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem
    shapes = [(256, 1024, 4096), (130, 512, 1024), (45, 2048, 2048)]
    prob = DeviceProblem(workloads.make_groups(shapes, seed=81))
    cap = torch.cuda.Stream()
    with gemm_env(kind):
        prob.step()
        torch.cuda.synchronize()
        with torch.cuda.stream(cap):
            prob.step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            prob.step()
    o = oracle.get()
    for rep in range(3):
        groups = workloads.make_groups(shapes, seed=200 + rep)
        for i, gr in enumerate(groups):
            prob.A[i].copy_(torch.from_numpy(np.ascontiguousarray(gr.A).reshape(-1)))
            prob.B[i].copy_(torch.from_numpy(np.ascontiguousarray(gr.B).reshape(-1)))
            prob.SFA[i].copy_(torch.from_numpy(np.ascontiguousarray(gr.SFA).reshape(-1)))
            prob.SFB[i].copy_(torch.from_numpy(np.ascontiguousarray(gr.SFB).reshape(-1)))
        for c in prob.C:
            c.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for gr, c in zip(groups, prob.outputs_fp16_bits()):
            compare_fp16(c, o.gemm(gr.A, gr.SFA, gr.B, gr.SFB, gr.M, gr.N, gr.K), f"replay {rep}")


def test_plan_picks_by_shape_class():
    """The configuration the library picks per shape class on this GPU: CTA
    pairs for the 4096^3 groups and for calls of fewer tiles than SMs, 128 x
    256 tiles for the small-M MoE shapes, 128 x 128 tiles for calls that fit
    one round of the grid in them and when some N of a larger call is not a
    multiple of 256; one launch per 32 groups."""
    from block_scaled_nvfp4_group_gb300 import ops, workloads
    from block_scaled_nvfp4_group_gb300.device import DeviceProblem

    def plan(groups):
        return ops.group_gemm_plan(descs=DeviceProblem(groups).descs)

    assert plan(workloads.make_workload("square").groups) == ("pair", 1)
    assert plan(workloads.make_workload("moe_gate_up").groups) == ("wide", 1)
    assert plan(workloads.make_workload("moe_down").groups) == ("wide", 1)
    assert plan(workloads.make_workload("quantized").groups) == ("pair", 1)
    assert plan(workloads.make_workload("tiny").groups) == ("compute", 1)
    assert plan(workloads.make_groups([(300, 264, 256)], seed=1)) == ("compute", 1)
    assert plan(workloads.make_groups([(300, 264, 256)] * 60, seed=1)) == ("stream", 2)
    shapes = [(64, 256, 256)] * 40
    assert plan(workloads.make_groups(shapes, seed=1)) == ("compute", 2)


@pytest.mark.parametrize("shape", [(1, 1 << 20, 256), (1 << 20, 256, 256), (256, 256, 1 << 20)])
def test_maximum_dimensions(shape):
    """Each of M, N, K at the documented maximum (2^20): tile and stage
    counts, relayout items and tensor-map coordinates at their largest;
    sampled rows against the oracle (the 2^20-row case runs on CTA pairs)."""
    from block_scaled_nvfp4_group_gb300 import workloads
    groups = workloads.make_groups([shape], seed=91)
    M, N, K = shape
    if K == 1 << 20:
        # an FP32 sum of 2^20 random products drifts past the tolerance the
        # workloads' K <= 7168 are held to; keep 64 random 16-element scale
        # blocks per row of A (the rest zero), so every K position is still
        # loaded and addressed but each output sums ~1000 products, and a
        # wrong K offset would move the non-zero blocks
        rng = np.random.default_rng(92)
        keep = np.zeros_like(groups[0].SFA)
        for r in range(M):
            idx = rng.choice(K // 16, size=64, replace=False)
            keep[r, idx] = groups[0].SFA[r, idx]
        groups[0].SFA[...] = keep
    run_and_compare(groups, rows_per_group=4, seed=9)
    torch.cuda.empty_cache()
