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


_FIRST_CALL_SCRIPT = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from block_scaled_nvfp4_group_gb300 import _abi, workloads
from oracle import oracle
lib = _abi.load()
o = oracle.get()
torch.cuda.init()
shapes = [(130, 264, 512), (64, 256, 256)]
groups = workloads.make_groups(shapes, seed=33)
keep, descs = [], (_abi.GroupDesc * len(groups))()
for i, g in enumerate(groups):
    # tiled scales made on the host, so that no other library call precedes
    sa = torch.from_numpy(o.sf_relayout(g.SFA, g.M, g.K)).cuda()
    sb = torch.from_numpy(o.sf_relayout(g.SFB, g.N, g.K)).cuda()
    A = torch.from_numpy(g.A).cuda().reshape(-1)
    B = torch.from_numpy(g.B).cuda().reshape(-1)
    C = torch.full((g.M, g.N), float("nan"), dtype=torch.float16, device="cuda")
    keep.append((A, B, sa, sb, C))
    descs[i] = _abi.GroupDesc(A.data_ptr(), B.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(),
                              g.M, g.N, g.K)
torch.cuda.synchronize()
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
free = []
for call in range(2):
    rc = lib.nvfp4_group_gemm_noalloc(descs, len(groups), stream)
    assert rc == _abi.NVFP4_OK, rc
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
print("FREE", free[0], free[1])
for g, (_, _, _, _, C) in zip(groups, keep):
    ref = o.gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K).view(np.float16).astype(np.float64)
    got = C.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-3 * np.abs(ref) + 1e-2), "mismatch"
print("FIRST_CALL_OK")
"""


def test_noalloc_as_first_library_call_in_a_fresh_process():
    """In a process whose first library call is the no-allocation entry
    point (tiled scales prepared on the host), the output equals the
    oracle's, and a second call leaves the device's free memory unchanged."""
    require_gb300()
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_SCRIPT, root], capture_output=True, text=True,
                       timeout=600, cwd=root)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "FIRST_CALL_OK" in r.stdout
    free = [int(x) for x in next(ln for ln in r.stdout.splitlines() if ln.startswith("FREE")).split()[1:]]
    assert free[0] == free[1], free
