"""ctypes declarations of the C ABI in include/nvfp4_group_gemm.h.

Argument marshalling only: every step of the computation runs in the CUDA
library.  Loading fails loudly when the library has not been built; there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libnvfp4_group_gemm.so")

NVFP4_OK = 0
NVFP4_ERR_INVALID_ARGUMENT = -1
NVFP4_ERR_MISALIGNED = -2
NVFP4_ERR_UNSUPPORTED = -3
NVFP4_ERR_CUDA = -4
NVFP4_ERR_TIMEOUT = -5
NVFP4_ERR_TOO_MANY = -6

# kernel configurations (NVFP4_KIND_* in the header) and their kernels
KIND_NAMES = {0: "stream", 1: "wide", 2: "compute", 3: "wide512", 4: "wide_p2", 5: "wide_p4",
              6: "pair", 7: "wide_sk", 8: "swap"}
KIND_KERNELS = {k: ("nvfp4_group_gemm_pair_kernel" if k == 6 else
                    "nvfp4_group_gemm_swap_kernel" if k == 8 else "nvfp4_group_gemm_kernel")
                for k in KIND_NAMES}


class GroupDesc(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("SFA", ctypes.c_void_p),
                ("SFB", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int)]


class GemmEpilogue(ctypes.Structure):
    _fields_ = [("alpha", ctypes.POINTER(ctypes.c_float)), ("out_bf16", ctypes.c_int),
                ("swiglu", ctypes.c_int)]


class SfRelayoutDesc(ctypes.Structure):
    _fields_ = [("src", ctypes.c_void_p), ("dst", ctypes.c_void_p),
                ("rows", ctypes.c_int), ("K", ctypes.c_int)]


class StepDesc(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("SFA", ctypes.c_void_p),
                ("SFB", ctypes.c_void_p), ("SFA_tiled", ctypes.c_void_p),
                ("SFB_tiled", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int)]


# name -> (restype, argtypes); every symbol declared in the header
SIGNATURES = {
    "nvfp4_group_gemm": (ctypes.c_int, [ctypes.POINTER(GroupDesc), ctypes.c_int, ctypes.c_void_p]),
    "nvfp4_group_gemm_noalloc": (ctypes.c_int, [ctypes.POINTER(GroupDesc), ctypes.c_int,
                                                ctypes.c_void_p]),
    "nvfp4_group_gemm_ex": (ctypes.c_int, [ctypes.POINTER(GroupDesc), ctypes.c_int,
                                           ctypes.POINTER(GemmEpilogue), ctypes.c_void_p]),
    "nvfp4_group_gemm_plan": (ctypes.c_int, [ctypes.POINTER(GroupDesc), ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_int)]),
    "nvfp4_group_gemm_plan_for": (ctypes.c_int, [ctypes.POINTER(GroupDesc), ctypes.c_int, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_int),
                                                 ctypes.POINTER(ctypes.c_int)]),
    "nvfp4_sf_relayout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_void_p]),
    "nvfp4_sf_relayout_group": (ctypes.c_int, [ctypes.POINTER(SfRelayoutDesc), ctypes.c_int,
                                               ctypes.c_void_p]),
    "nvfp4_sf_tiled_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int]),
    "nvfp4_relayout_and_gemm": (ctypes.c_int, [ctypes.POINTER(StepDesc), ctypes.c_int,
                                               ctypes.POINTER(GemmEpilogue), ctypes.c_void_p]),
    "nvfp4_quantize": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p]),
    "nvfp4_last_device_error": (ctypes.c_int, [ctypes.c_void_p]),
    "nvfp4_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "nvfp4_debug_drop_first_stage": (None, [ctypes.c_int]),
    "nvfp4_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "nvfp4_version": (ctypes.c_int, []),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (built by __graft_entry__.build() or
    block_scaled_nvfp4_group_gb300/build.py)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"NVFP4 CUDA library not built: {path} is missing "
                          "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


class Nvfp4Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = load().nvfp4_strerror(code).decode()
        super().__init__(f"{what}: {msg} ({code})")


def check(code: int, what: str) -> None:
    if code != NVFP4_OK:
        raise Nvfp4Error(code, what)
