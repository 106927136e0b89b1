"""PyTorch-facing wrappers of the C ABI (argument marshalling only).

Tensors provide device memory and the current CUDA stream; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback:
without the built library, or without a GB300, these calls raise.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi


def _stream_handle(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_device(t: torch.Tensor, name: str) -> None:
    """The library works on the current CUDA device: every buffer it is
    given must live there (a host or another GPU's pointer would fault)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")


def _check_u8(t: torch.Tensor, name: str, numel: int) -> None:
    _check_device(t, name)
    if t.dtype not in (torch.uint8, torch.int8) and t.element_size() != 1:
        raise ValueError(f"{name} must hold bytes (uint8), got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} bytes, expected {numel}")


def sf_tiled_bytes(rows: int, K: int) -> int:
    return int(_abi.load().nvfp4_sf_tiled_bytes(rows, K))


def sf_relayout(sf: torch.Tensor, rows: int, K: int, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """Row-major [rows, K/16] E4M3FN scales (uint8) -> tiled layout (uint8)."""
    lib = _abi.load()
    _check_u8(sf, "sf", rows * K // 16)
    nbytes = sf_tiled_bytes(rows, K)
    if out is None:
        out = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=sf.device)
    else:
        _check_device(out, "out")
        if out.numel() * out.element_size() < nbytes:
            raise ValueError("out too small")
    _abi.check(lib.nvfp4_sf_relayout(ctypes.c_void_p(sf.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                     rows, K, _stream_handle(stream)), "nvfp4_sf_relayout")
    return out


def make_relayout_descs(items):
    """items: iterable of (src, dst, rows, K) device tensors."""
    items = list(items)
    arr = (_abi.SfRelayoutDesc * len(items))()
    for i, (src, dst, rows, K) in enumerate(items):
        _check_u8(src, "src", rows * K // 16)
        _check_device(dst, "dst")
        if dst.numel() * dst.element_size() < sf_tiled_bytes(rows, K):
            raise ValueError("dst too small")
        arr[i] = _abi.SfRelayoutDesc(src.data_ptr(), dst.data_ptr(), rows, K)
    return arr


def sf_relayout_group(items, stream=None, descs=None) -> None:
    """items: iterable of (src, dst, rows, K) device tensors; one launch.
    `descs` may carry a prebuilt array (make_relayout_descs)."""
    lib = _abi.load()
    arr = descs if descs is not None else make_relayout_descs(items)
    if len(arr) == 0:
        return
    _abi.check(lib.nvfp4_sf_relayout_group(arr, len(arr), _stream_handle(stream)),
               "nvfp4_sf_relayout_group")


def make_group_descs(groups, out_bf16: bool = False, swiglu: bool = False):
    """groups: iterable of (A, B, SFA_tiled, SFB_tiled, C, M, N, K); C is
    [M, N] float16, or as the fused epilogue writes it (bfloat16, [M, N/2])."""
    groups = list(groups)
    arr = (_abi.GroupDesc * len(groups))()
    for i, (A, B, SFA, SFB, C, M, N, K) in enumerate(groups):
        if M > 0:
            _check_u8(A, "A", M * K // 2)
            _check_u8(B, "B", N * K // 2)
            _check_device(SFA, "SFA (tiled)")
            _check_device(SFB, "SFB (tiled)")
            _check_device(C, "C")
            if (SFA.numel() * SFA.element_size() < sf_tiled_bytes(M, K) or
                    SFB.numel() * SFB.element_size() < sf_tiled_bytes(N, K)):
                raise ValueError("scale buffers too small")
            want = torch.bfloat16 if out_bf16 else torch.float16
            n_out = N // 2 if swiglu else N
            if C.dtype != want or C.numel() != M * n_out or not C.is_contiguous():
                raise ValueError(f"C must be a contiguous {want} [M, {n_out}] tensor")
        arr[i] = _abi.GroupDesc(A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                                C.data_ptr(), M, N, K)
    return arr


def group_gemm(groups, stream=None, descs=None) -> None:
    """C_g = A_g . B_g^T for every group (see include/nvfp4_group_gemm.h).
    groups: iterable of (A, B, SFA_tiled, SFB_tiled, C, M, N, K) with device
    tensors; C is overwritten.  `descs` may carry a prebuilt descriptor array
    (make_group_descs) to skip the per-call marshalling."""
    lib = _abi.load()
    arr = descs if descs is not None else make_group_descs(groups)
    _abi.check(lib.nvfp4_group_gemm(arr, len(arr), _stream_handle(stream)), "nvfp4_group_gemm")


def group_gemm_ex(groups, alpha=None, out_bf16: bool = False, swiglu: bool = False, stream=None,
                  descs=None) -> None:
    """group_gemm with the fused epilogue (nvfp4_group_gemm_ex): per-group
    scales `alpha` (sequence of floats or None), BF16 output, SwiGLU of
    128-row gate / up blocks (C is then [M, N/2])."""
    lib = _abi.load()
    arr = descs if descs is not None else make_group_descs(groups, out_bf16=out_bf16, swiglu=swiglu)
    epi = _abi.GemmEpilogue()
    keep = None
    if alpha is not None:
        keep = (ctypes.c_float * len(arr))(*[float(a) for a in alpha])
        epi.alpha = ctypes.cast(keep, ctypes.POINTER(ctypes.c_float))
    epi.out_bf16 = 1 if out_bf16 else 0
    epi.swiglu = 1 if swiglu else 0
    _abi.check(lib.nvfp4_group_gemm_ex(arr, len(arr), ctypes.byref(epi), _stream_handle(stream)),
               "nvfp4_group_gemm_ex")
    del keep


def make_step_descs(steps, out_bf16: bool = False, swiglu: bool = False):
    """steps: iterable of (A, B, SFA, SFB, SFA_tiled, SFB_tiled, C, M, N, K)
    device tensors, SFA / SFB the row-major scales [M, K/16] / [N, K/16]."""
    steps = list(steps)
    arr = (_abi.StepDesc * len(steps))()
    checked = make_group_descs([(A, B, SFA_t, SFB_t, C, M, N, K)
                                for (A, B, SFA, SFB, SFA_t, SFB_t, C, M, N, K) in steps],
                               out_bf16=out_bf16, swiglu=swiglu)
    for i, (A, B, SFA, SFB, SFA_t, SFB_t, C, M, N, K) in enumerate(steps):
        if M > 0:
            _check_u8(SFA, "SFA", M * K // 16)
            _check_u8(SFB, "SFB", N * K // 16)
        g = checked[i]
        arr[i] = _abi.StepDesc(g.A, g.B, SFA.data_ptr() if M > 0 else None,
                               SFB.data_ptr() if M > 0 else None, g.SFA, g.SFB, g.C, M, N, K)
    return arr


def relayout_and_gemm(steps=None, alpha=None, out_bf16: bool = False, swiglu: bool = False,
                      stream=None, descs=None) -> None:
    """The whole path of one grouped call (nvfp4_relayout_and_gemm): the
    relayout of every SFA / SFB into the tiled buffers, then the grouped GEMM
    (fused epilogue options as group_gemm_ex)."""
    lib = _abi.load()
    arr = descs if descs is not None else make_step_descs(steps, out_bf16=out_bf16, swiglu=swiglu)
    epi = _abi.GemmEpilogue()
    keep = None
    if alpha is not None:
        keep = (ctypes.c_float * len(arr))(*[float(a) for a in alpha])
        epi.alpha = ctypes.cast(keep, ctypes.POINTER(ctypes.c_float))
    epi.out_bf16 = 1 if out_bf16 else 0
    epi.swiglu = 1 if swiglu else 0
    _abi.check(lib.nvfp4_relayout_and_gemm(arr, len(arr), ctypes.byref(epi), _stream_handle(stream)),
               "nvfp4_relayout_and_gemm")
    del keep


def group_gemm_plan(groups=None, descs=None):
    """(kind name, launches) nvfp4_group_gemm would use for these groups on
    the current device; nothing is launched."""
    lib = _abi.load()
    arr = descs if descs is not None else make_group_descs(groups)
    kind, launches = ctypes.c_int(-1), ctypes.c_int(0)
    _abi.check(lib.nvfp4_group_gemm_plan(arr, len(arr), ctypes.byref(kind), ctypes.byref(launches)),
               "nvfp4_group_gemm_plan")
    return _abi.KIND_NAMES[kind.value], launches.value


def group_gemm_plan_for(descs, sm_count: int):
    """(kind name, launches) for a device with `sm_count` SMs, computed on the
    host alone (no GPU needed); `descs` is a GroupDesc array."""
    lib = _abi.load()
    kind, launches = ctypes.c_int(-1), ctypes.c_int(0)
    _abi.check(lib.nvfp4_group_gemm_plan_for(descs, len(descs), sm_count, ctypes.byref(kind),
                                             ctypes.byref(launches)),
               "nvfp4_group_gemm_plan_for")
    return _abi.KIND_NAMES[kind.value], launches.value


def quantize(x: torch.Tensor, codes: torch.Tensor | None = None, sf_tiled: torch.Tensor | None = None,
             sf_rowmajor: torch.Tensor | None = None, want_rowmajor: bool = False, stream=None):
    """NVFP4 quantisation of a [rows, K] float16 / bfloat16 CUDA tensor (see
    nvfp4_quantize): returns (codes uint8 [rows, K/2], tiled scales uint8,
    row-major scales uint8 [rows, K/16] or None)."""
    if x.dtype not in (torch.float16, torch.bfloat16) or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D float16 or bfloat16 tensor")
    _check_device(x, "x")
    rows, K = x.shape
    if codes is None:
        codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device)
    else:
        _check_u8(codes, "codes", rows * K // 2)
    if sf_tiled is None:
        sf_tiled = torch.empty(max(sf_tiled_bytes(rows, K), 16), dtype=torch.uint8, device=x.device)
    else:
        _check_device(sf_tiled, "sf_tiled")
        if sf_tiled.numel() * sf_tiled.element_size() < sf_tiled_bytes(rows, K):
            raise ValueError("sf_tiled too small")
    if sf_rowmajor is None and want_rowmajor:
        sf_rowmajor = torch.empty((rows, K // 16), dtype=torch.uint8, device=x.device)
    elif sf_rowmajor is not None:
        _check_u8(sf_rowmajor, "sf_rowmajor", rows * K // 16)
    lib = _abi.load()
    _abi.check(lib.nvfp4_quantize(x.data_ptr(), 1 if x.dtype == torch.bfloat16 else 0, rows, K,
                                  codes.data_ptr(), sf_tiled.data_ptr(),
                                  sf_rowmajor.data_ptr() if sf_rowmajor is not None else None,
                                  _stream_handle(stream)), "nvfp4_quantize")
    return codes, sf_tiled, sf_rowmajor


def last_device_error(stream=None) -> int:
    return int(_abi.load().nvfp4_last_device_error(_stream_handle(stream)))


def set_wait_timeout_ns(ns: int) -> None:
    _abi.load().nvfp4_set_wait_timeout_ns(int(ns))


def debug_drop_first_stage(enable: bool) -> None:
    _abi.load().nvfp4_debug_drop_first_stage(1 if enable else 0)
