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
