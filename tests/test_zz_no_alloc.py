"""nvfp4_group_gemm_noalloc: the grouped GEMM for callers that may not
allocate device memory (engines whose device memory is all planned ahead
and handed to them, latency-critical loops that cannot take an
allocation's synchronisation).  It keeps the kernel's status words in a
static array inside the library instead of allocating them.

Checked here through the C ABI: its output equals the output of
nvfp4_group_gemm within the tolerance of the parity tests, on two calls in
a row (the second call must overwrite C and reuse the static array), for a
single launch and for a call split into two launches; and a call needing
more than the array holds is refused without a launch.  This file is
collected last so that a failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import compare_fp16, require_gb300

pytestmark = pytest.mark.gpu


def _problem(shapes, seed):
    from block_scaled_nvfp4_group_gb300 import ops, workloads
    groups = workloads.make_groups(shapes, seed=seed)
    keep, descs_ref, descs_na, outs = [], [], [], []
    for g in groups:
        A = torch.from_numpy(g.A).cuda().reshape(-1)
        B = torch.from_numpy(g.B).cuda().reshape(-1)
        if g.M > 0:
            sa = ops.sf_relayout(torch.from_numpy(g.SFA).cuda().reshape(-1), g.M, g.K)
            sb = ops.sf_relayout(torch.from_numpy(g.SFB).cuda().reshape(-1), g.N, g.K)
        else:
            sa = sb = torch.zeros(16, dtype=torch.uint8, device="cuda")
        c_ref = torch.empty((g.M, g.N), dtype=torch.float16, device="cuda")
        c_na = torch.empty((g.M, g.N), dtype=torch.float16, device="cuda")
        keep += [A, B, sa, sb]
        descs_ref.append((A, B, sa, sb, c_ref, g.M, g.N, g.K))
        descs_na.append((A, B, sa, sb, c_na, g.M, g.N, g.K))
        outs.append((c_ref, c_na))
    return keep, descs_ref, descs_na, outs


def _check_against_group_gemm(shapes, seed):
    from block_scaled_nvfp4_group_gb300 import _abi, ops
    lib = _abi.load()
    keep, descs_ref, descs_na, outs = _problem(shapes, seed)
    ops.group_gemm(descs_ref)                       # the existing entry point
    arr = ops.make_group_descs(descs_na)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        for _, c_na in outs:
            c_na.fill_(float("nan"))                # every element must be rewritten
        rc = lib.nvfp4_group_gemm_noalloc(arr, len(arr), stream)
        assert rc == _abi.NVFP4_OK, lib.nvfp4_strerror(rc)
        torch.cuda.synchronize()
        for i, (c_ref, c_na) in enumerate(outs):
            if c_ref.numel() == 0:
                continue
            compare_fp16(c_na.view(torch.int16).cpu().numpy().view(np.uint16),
                         c_ref.view(torch.int16).cpu().numpy().view(np.uint16),
                         f"call {call} group {i}")
    del keep


def test_noalloc_matches_group_gemm_one_launch():
    require_gb300()
    _check_against_group_gemm([(200, 384, 1024), (77, 256, 512), (0, 256, 256),
                               (300, 520, 768), (1, 8, 256)], seed=31)


def test_noalloc_matches_group_gemm_two_launches():
    require_gb300()
    rng = np.random.default_rng(32)
    shapes = [(int(rng.integers(1, 150)), 8 * int(rng.integers(1, 30)), 256 * int(rng.integers(1, 3)))
              for _ in range(40)]                   # 40 groups: two launches, two status slots
    _check_against_group_gemm(shapes, seed=32)


def test_noalloc_refuses_more_than_its_scratch_holds():
    require_gb300()
    from block_scaled_nvfp4_group_gb300 import _abi
    lib = _abi.load()
    n = 32 * 32 + 1                                 # one group more than 32 launches take
    arr = (_abi.GroupDesc * n)(*[_abi.GroupDesc(256, 256, 256, 256, 256, 1, 8, 256)
                                 for _ in range(n)])
    assert lib.nvfp4_group_gemm_noalloc(arr, n, None) == _abi.NVFP4_ERR_TOO_MANY
