"""The C-ABI library builds, loads and exports every symbol its header
declares; argument validation rejects bad calls before touching the GPU.
(No compute call: these run on machines without a GPU.)"""
import ctypes
import os
import re

import pytest

from block_scaled_nvfp4_group_gb300 import _abi, build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4_group_gemm.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _abi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("nvfp4_group_gemm", "nvfp4_sf_relayout", "nvfp4_sf_relayout_group",
                 "nvfp4_sf_tiled_bytes", "nvfp4_last_device_error", "nvfp4_strerror"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _abi.SIGNATURES, f"{name} missing from the Python binding"
    assert set(_abi.SIGNATURES) == set(declared_functions())


def test_struct_layouts_match_header():
    # GroupDesc: 5 pointers + 3 ints (+ 4 bytes tail padding on LP64)
    assert ctypes.sizeof(_abi.GroupDesc) == 5 * 8 + 3 * 4 + 4
    assert ctypes.sizeof(_abi.SfRelayoutDesc) == 2 * 8 + 2 * 4
    # StepDesc: 7 pointers + 3 ints (+ 4 bytes tail padding)
    assert ctypes.sizeof(_abi.StepDesc) == 7 * 8 + 3 * 4 + 4


def test_strerror_and_version(lib):
    for code in range(-7, 1):
        assert lib.nvfp4_strerror(code)
    assert lib.nvfp4_version() >= (0 << 16) | (1 << 8)


def test_tiled_bytes(lib):
    assert lib.nvfp4_sf_tiled_bytes(1, 256) == 4 * 512
    assert lib.nvfp4_sf_tiled_bytes(128, 256) == 4 * 512
    assert lib.nvfp4_sf_tiled_bytes(129, 7168) == 2 * 112 * 512
    assert lib.nvfp4_sf_tiled_bytes(0, 256) == 0
    assert lib.nvfp4_sf_tiled_bytes(5, 100) == 0


def _desc(A=16, B=16, SFA=16, SFB=16, C=16, M=128, N=128, K=256):
    return _abi.GroupDesc(A, B, SFA, SFB, C, M, N, K)


@pytest.mark.parametrize("desc,code", [
    (dict(K=100), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    (dict(K=384), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    (dict(N=12), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    (dict(N=0), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    (dict(M=-1), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    (dict(M=1 << 21), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    (dict(A=0), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    (dict(C=0), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    (dict(A=24), _abi.NVFP4_ERR_MISALIGNED),
    (dict(SFB=8), _abi.NVFP4_ERR_MISALIGNED),
    (dict(C=2), _abi.NVFP4_ERR_MISALIGNED),
])
def test_group_gemm_rejects_before_launch(lib, desc, code):
    arr = (_abi.GroupDesc * 2)(_desc(), _desc(**desc))
    assert lib.nvfp4_group_gemm(arr, 2, None) == code


def test_group_gemm_count_limits(lib):
    arr = (_abi.GroupDesc * 1)(_desc())
    assert lib.nvfp4_group_gemm(arr, 0, None) == _abi.NVFP4_ERR_INVALID_ARGUMENT
    assert lib.nvfp4_group_gemm(None, 1, None) == _abi.NVFP4_ERR_INVALID_ARGUMENT
    big = (_abi.GroupDesc * 4097)()
    assert lib.nvfp4_group_gemm(big, 4097, None) == _abi.NVFP4_ERR_TOO_MANY


@pytest.mark.parametrize("args,code", [
    ((16, 16, 10, 100), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    ((16, 16, -1, 256), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    ((0, 16, 10, 256), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    ((16, 0, 10, 256), _abi.NVFP4_ERR_INVALID_ARGUMENT),
    ((17, 16, 10, 256), _abi.NVFP4_ERR_MISALIGNED),
    ((16, 20, 10, 256), _abi.NVFP4_ERR_MISALIGNED),
])
def test_relayout_rejects_before_launch(lib, args, code):
    assert lib.nvfp4_sf_relayout(*args, None) == code
    arr = (_abi.SfRelayoutDesc * 1)(_abi.SfRelayoutDesc(*args))
    assert lib.nvfp4_sf_relayout_group(arr, 1, None) == code


P = 16   # a 16-byte-aligned stand-in address: validation never dereferences it


def _step(a=P, sfa=P, **kw):
    d = dict(A=a, B=P, SFA=sfa, SFB=P, SFA_tiled=P, SFB_tiled=P, C=P, M=128, N=256, K=256)
    d.update(kw)
    return _abi.StepDesc(d["A"], d["B"], d["SFA"], d["SFB"], d["SFA_tiled"], d["SFB_tiled"], d["C"],
                         d["M"], d["N"], d["K"])


@pytest.mark.parametrize("step,code", [
    (_step(sfa=None), _abi.NVFP4_ERR_INVALID_ARGUMENT),          # no row-major scales
    (_step(sfa=P + 4), _abi.NVFP4_ERR_MISALIGNED),
    (_step(K=320), _abi.NVFP4_ERR_INVALID_ARGUMENT),             # K % 256 != 0
    (_step(SFA_tiled=None), _abi.NVFP4_ERR_INVALID_ARGUMENT),    # no tiled buffer
    (_step(a=P + 8), _abi.NVFP4_ERR_MISALIGNED),
])
def test_relayout_and_gemm_rejects_before_launch(lib, step, code):
    arr = (_abi.StepDesc * 1)(step)
    assert lib.nvfp4_relayout_and_gemm(arr, 1, None, None) == code
    assert lib.nvfp4_relayout_and_gemm(None, 1, None, None) == _abi.NVFP4_ERR_INVALID_ARGUMENT
    assert lib.nvfp4_relayout_and_gemm(arr, 0, None, None) == _abi.NVFP4_ERR_INVALID_ARGUMENT


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        _abi.load(str(tmp_path / "missing.so"))


# --- the host plan: kernel configuration and launch count, no GPU --------

MOE_M = [366, 261, 336, 45, 223, 107, 317, 349]


def _plan(lib, shapes, sm=152):
    arr = (_abi.GroupDesc * len(shapes))(*[_desc(M=m, N=n, K=k) for m, n, k in shapes])
    kind, launches = ctypes.c_int(-1), ctypes.c_int(-1)
    rc = lib.nvfp4_group_gemm_plan_for(arr, len(arr), sm, ctypes.byref(kind), ctypes.byref(launches))
    return rc, _abi.KIND_NAMES.get(kind.value), launches.value


@pytest.mark.parametrize("shapes,sm,kind,launches", [
    # small-M MoE shapes, every N a multiple of 256: 128 x 256 tiles (pairs
    # would pad M to 256 rows and add a round of the grid)
    ([(m, 4096, 7168) for m in MOE_M], 152, "wide", 1),
    ([(m, 7168, 2048) for m in MOE_M], 152, "wide", 1),
    ([(64, 4096, 7168)] * 8, 152, "wide", 1),
    # 2048 tiles of 128 x 256 = 14 rounds of 152; 1024 pair tiles = 14 rounds of 76
    ([(4096, 4096, 4096)] * 4, 152, "pair", 1),
    # fewer tiles than SMs: pairs need no more rounds (1 = 1) ...
    ([(512, 3072, 4096)] * 2, 152, "pair", 1),
    ([(1000, 4096, 2048)] * 2, 152, "pair", 1),
    # ... and the same on 8 SMs (12 = 12 rounds)
    ([(512, 3072, 4096)] * 2, 8, "pair", 1),
    # 768 tiles = 6 rounds, 512 pair tiles = 7 rounds of 76: pairing would add one
    ([(384, 4096, 256)] * 16, 152, "wide", 1),
    # 128 x 128 tiles that fit one round of the grid
    ([(64, 256, 256), (128, 256, 256)], 152, "compute", 1),
    ([(256, 2048, 2048)] * 4, 152, "compute", 1),
    ([(300, 1024, 1024)] * 6, 152, "compute", 1),
    ([(77, 136, 512)], 152, "compute", 1),
    # ... up to exactly one round (152 tiles of 128 x 128) but not past it
    # (154, 160): then 128 x 256 tiles, since pairs would need two rounds
    ([(128, 256, 256)] * 76, 152, "compute", 3),
    ([(128, 256, 256)] * 77, 152, "wide", 3),
    ([(128, 256, 256)] * 80, 152, "wide", 3),
    # SM count of the plan: the same call on 8 SMs is many rounds of pairs
    ([(256, 2048, 2048)] * 4, 8, "pair", 1),
    # one N off the 256 grid sends a larger call to 128-column tiles
    ([(4096, 4096, 4096), (64, 136, 256)], 152, "stream", 1),
    ([(300, 264, 4096)] * 60, 152, "stream", 2),
    # 32 groups per launch; empty groups take no slot
    ([(64, 256, 256)] * 32, 152, "compute", 1),
    ([(64, 256, 256)] * 33, 152, "compute", 2),
    ([(64, 256, 256)] * 65, 152, "compute", 3),
    ([(0, 256, 256)] * 40 + [(64, 256, 256)] * 30, 152, "compute", 1),
    ([(0, 256, 256)] * 3, 152, "compute", 0),
])
def test_plan_kind_and_launches(lib, monkeypatch, shapes, sm, kind, launches):
    monkeypatch.delenv("NVFP4_GEMM_KIND", raising=False)
    assert _plan(lib, shapes, sm) == (_abi.NVFP4_OK, kind, launches)


@pytest.mark.parametrize("forced,shapes,kind", [
    ("0", [(m, 4096, 7168) for m in MOE_M], "stream"),
    ("7", [(m, 4096, 7168) for m in MOE_M], "wide_sk"),
    ("6", [(m, 4096, 7168) for m in MOE_M], "pair"),
    ("1", [(m, 4096, 7168) for m in MOE_M], "wide"),
    ("8", [(4096, 4096, 256)], "swap"),
    ("8", [(m, 4096, 7168) for m in MOE_M], "swap"),
    # the swapped kernel takes any N (rows of B past N load as zeros)
    ("8", [(77, 136, 512)], "swap"),
    ("1", [(4096, 4096, 4096)] * 4, "wide"),
    # a forced kind that cannot take the shapes falls back to 128-column tiles
    ("1", [(77, 136, 512)], "stream"),
    ("6", [(64, 128, 256)], "stream"),
    ("7", [(77, 136, 512)], "stream"),
    # out of range: ignored
    ("99", [(4096, 4096, 4096)] * 4, "pair"),
])
def test_plan_forced_kind(lib, monkeypatch, forced, shapes, kind):
    monkeypatch.setenv("NVFP4_GEMM_KIND", forced)
    rc, k, n = _plan(lib, shapes)
    assert (rc, k) == (_abi.NVFP4_OK, kind)
    assert n == 1


def test_plan_swap_token_tiles_across_launches(lib, monkeypatch):
    # 4096 rows = 16 token tiles per group: 4 groups fill two launches of 32
    # token tiles; a group's tiles may continue in the next launch; a swap
    # launch takes 16 groups and 32 token tiles, empty groups take no slot
    monkeypatch.setenv("NVFP4_GEMM_KIND", "8")
    assert _plan(lib, [(64, 256, 256)] * 16) == (_abi.NVFP4_OK, "swap", 1)
    assert _plan(lib, [(64, 256, 256)] * 17) == (_abi.NVFP4_OK, "swap", 2)
    assert _plan(lib, [(300, 256, 256)] * 17) == (_abi.NVFP4_OK, "swap", 2)
    assert _plan(lib, [(0, 256, 256)] * 40 + [(64, 256, 256)] * 30) == (_abi.NVFP4_OK, "swap", 2)
    assert _plan(lib, [(384, 4096, 256)] * 16) == (_abi.NVFP4_OK, "swap", 1)
    assert _plan(lib, [(4096, 4096, 4096)] * 4) == (_abi.NVFP4_OK, "swap", 2)
    assert _plan(lib, [(4096, 4096, 4096)] * 4 + [(1, 256, 256)]) == (_abi.NVFP4_OK, "swap", 3)
    assert _plan(lib, [(2 << 18, 256, 256)]) == (_abi.NVFP4_OK, "swap", 64)


def test_plan_pair_launch_counts_256_row_tiles(lib, monkeypatch):
    # launch splitting counts tiles of the chosen kind: 33 groups still need
    # two launches with pair tiles
    monkeypatch.setenv("NVFP4_GEMM_KIND", "6")
    assert _plan(lib, [(512, 256, 256)] * 33) == (_abi.NVFP4_OK, "pair", 2)


def test_plan_rejects_before_anything(lib):
    kind, launches = ctypes.c_int(-5), ctypes.c_int(-5)
    arr = (_abi.GroupDesc * 1)(_desc())
    assert lib.nvfp4_group_gemm_plan_for(arr, 1, 1, ctypes.byref(kind), ctypes.byref(launches)) == \
        _abi.NVFP4_ERR_INVALID_ARGUMENT
    assert lib.nvfp4_group_gemm_plan_for(arr, 1, 152, None, ctypes.byref(launches)) == \
        _abi.NVFP4_ERR_INVALID_ARGUMENT
    bad = (_abi.GroupDesc * 1)(_desc(K=100))
    assert lib.nvfp4_group_gemm_plan_for(bad, 1, 152, ctypes.byref(kind), ctypes.byref(launches)) == \
        _abi.NVFP4_ERR_INVALID_ARGUMENT
    assert lib.nvfp4_group_gemm_plan_for(arr, 0, 152, ctypes.byref(kind), ctypes.byref(launches)) == \
        _abi.NVFP4_ERR_INVALID_ARGUMENT
    assert (kind.value, launches.value) == (-5, -5)     # written only on success


def test_binding_refuses_host_tensors(lib):
    """The Python layer marshals device tensors only: host tensors are refused
    before any library call, so nothing can run on a CPU copy."""
    import torch
    from block_scaled_nvfp4_group_gb300 import ops
    M, N, K = 128, 256, 256
    A = torch.zeros(M * K // 2, dtype=torch.uint8)
    B = torch.zeros(N * K // 2, dtype=torch.uint8)
    SFA = torch.zeros(ops.sf_tiled_bytes(M, K), dtype=torch.uint8)
    SFB = torch.zeros(ops.sf_tiled_bytes(N, K), dtype=torch.uint8)
    C = torch.zeros(M, N, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        ops.make_group_descs([(A, B, SFA, SFB, C, M, N, K)])
    with pytest.raises(ValueError, match="CUDA"):
        ops.make_relayout_descs([(torch.zeros(M * K // 16, dtype=torch.uint8), SFA, M, K)])
    with pytest.raises(ValueError, match="CUDA"):
        ops.sf_relayout(torch.zeros(M * K // 16, dtype=torch.uint8), M, K)
    with pytest.raises(ValueError, match="CUDA"):
        ops.quantize(torch.zeros(M, K, dtype=torch.float16))
