"""Python access to the CPU oracle (oracle/nvfp4_oracle.c).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module.  It shares no code with the CUDA path.

The oracle computes, for one group,
``C[m][n] = fp16_rne(sum_k e2m1(A[m][k]) * e4m3fn(SFA[m][k//16]) *
e2m1(B[n][k]) * e4m3fn(SFB[n][k//16]))`` in float64 (kernelbot
nvfp4-group-gemm submission 474067: header comment of the CUDA source and
``tcgen05_mma_nvfp4``, ``kind::mxf4nvf4.block_scale.block16``), with plain
row-major scale factors, defines the tiled scale-factor layout the GPU
kernel reads, and the NVFP4 quantisation that produces the operands
(per 16-block scale E4M3FN(absmax/6), codes E2M1(x/scale), decisions taken on
IEEE single-precision values).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "libnvfp4_oracle.so")

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)


def compile_oracle(src: str, out: str) -> str:
    """gcc, plain C11, -O2, pthreads; no contraction of a*b+c into FMA, so
    every product and every partial sum is rounded as written on every host
    architecture."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-pthread", "-D_DEFAULT_SOURCE", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(SOURCE), os.path.getmtime(__file__)):
        compile_oracle(SOURCE, _LIB)
    return _LIB


def _p(a, t):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(t)


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a))
    assert a.dtype == np.uint8, a.dtype
    return a


class Oracle:
    """Wrapper around one compiled copy of the oracle library."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        L.nvfp4_oracle_e2m1.restype = ctypes.c_double
        L.nvfp4_oracle_e2m1.argtypes = [ctypes.c_uint]
        L.nvfp4_oracle_e4m3fn.restype = ctypes.c_double
        L.nvfp4_oracle_e4m3fn.argtypes = [ctypes.c_uint]
        L.nvfp4_oracle_fp16_rne.restype = ctypes.c_uint16
        L.nvfp4_oracle_fp16_rne.argtypes = [ctypes.c_double]
        L.nvfp4_oracle_gemm.restype = ctypes.c_int
        L.nvfp4_oracle_gemm.argtypes = [_u8p, _u8p, _u8p, _u8p, _u16p, _f64p,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.nvfp4_oracle_gemm_rows.restype = ctypes.c_int
        L.nvfp4_oracle_gemm_rows.argtypes = [_u8p, _u8p, _u8p, _u8p, _u16p, _f64p,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             _i32p, ctypes.c_int, ctypes.c_int]
        L.nvfp4_oracle_gemm_elements.restype = ctypes.c_int
        L.nvfp4_oracle_gemm_elements.argtypes = [_u8p, _u8p, _u8p, _u8p,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 _i32p, _i32p, ctypes.c_int, _u16p]
        L.nvfp4_oracle_gemm_fixed.restype = ctypes.c_int
        L.nvfp4_oracle_gemm_fixed.argtypes = [_u8p, _u8p, _u8p, _u8p, _i64p,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.nvfp4_oracle_sf_tiled_bytes.restype = ctypes.c_size_t
        L.nvfp4_oracle_sf_tiled_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
        L.nvfp4_oracle_sf_relayout.restype = ctypes.c_int
        L.nvfp4_oracle_sf_relayout.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_int]
        L.nvfp4_oracle_sf_unrelayout.restype = ctypes.c_int
        L.nvfp4_oracle_sf_unrelayout.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_int]
        L.nvfp4_oracle_bf16_rne.restype = ctypes.c_uint16
        L.nvfp4_oracle_bf16_rne.argtypes = [ctypes.c_double]
        L.nvfp4_oracle_silu.restype = ctypes.c_double
        L.nvfp4_oracle_silu.argtypes = [ctypes.c_double]
        L.nvfp4_oracle_epilogue.restype = ctypes.c_int
        L.nvfp4_oracle_epilogue.argtypes = [_f64p, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                            ctypes.c_int, ctypes.c_int, _u16p]
        L.nvfp4_oracle_e4m3_rne.restype = ctypes.c_uint
        L.nvfp4_oracle_e4m3_rne.argtypes = [ctypes.c_float]
        L.nvfp4_oracle_e2m1_rne.restype = ctypes.c_uint
        L.nvfp4_oracle_e2m1_rne.argtypes = [ctypes.c_float]
        L.nvfp4_oracle_quantize.restype = ctypes.c_int
        L.nvfp4_oracle_quantize.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u8p, _u8p]
        self.L = L
        self.path = path

    # element decoders -----------------------------------------------------
    def e2m1(self, code: int) -> float:
        return self.L.nvfp4_oracle_e2m1(int(code))

    def e4m3fn(self, byte: int) -> float:
        return self.L.nvfp4_oracle_e4m3fn(int(byte))

    def fp16_rne_bits(self, x: float) -> int:
        return int(self.L.nvfp4_oracle_fp16_rne(float(x)))

    # one group --------------------------------------------------------------
    def gemm(self, A, SFA, B, SFB, M: int, N: int, K: int, rows=None, threads: int = 0,
             want_acc: bool = False):
        """A [M, K/2] u8, SFA [M, K/16] u8 (row-major), B [N, K/2],
        SFB [N, K/16].  Returns FP16 bits as uint16 [M, N] (only rows
        ``rows = (begin, end)`` computed when given, the rest zero), plus the
        float64 sums when ``want_acc``."""
        A, SFA, B, SFB = _u8(A), _u8(SFA), _u8(B), _u8(SFB)
        assert A.size == M * K // 2 and B.size == N * K // 2
        assert SFA.size == M * K // 16 and SFB.size == N * K // 16
        C = np.zeros((M, N), dtype=np.uint16)
        acc = np.zeros((M, N), dtype=np.float64) if want_acc else None
        r0, r1 = (0, M) if rows is None else rows
        rc = self.L.nvfp4_oracle_gemm(_p(A, _u8p), _p(SFA, _u8p), _p(B, _u8p), _p(SFB, _u8p),
                                      _p(C, _u16p), _p(acc, _f64p), M, N, K, r0, r1, threads)
        if rc != 0:
            raise ValueError(f"oracle gemm failed ({rc})")
        return (C, acc) if want_acc else C

    def gemm_rows(self, A, SFA, B, SFB, M: int, N: int, K: int, rows, threads: int = 0):
        """FP16 bits of the listed rows of C: uint16 [len(rows), N]."""
        A, SFA, B, SFB = _u8(A), _u8(SFA), _u8(B), _u8(SFB)
        assert A.size == M * K // 2 and B.size == N * K // 2
        assert SFA.size == M * K // 16 and SFB.size == N * K // 16
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        C = np.zeros((M, N), dtype=np.uint16)
        rc = self.L.nvfp4_oracle_gemm_rows(_p(A, _u8p), _p(SFA, _u8p), _p(B, _u8p), _p(SFB, _u8p),
                                           _p(C, _u16p), None, M, N, K, _p(rows, _i32p),
                                           rows.shape[0], threads)
        if rc != 0:
            raise ValueError(f"oracle gemm_rows failed ({rc})")
        return C[rows]

    def gemm_elements(self, A, SFA, B, SFB, M: int, N: int, K: int, ms, ns) -> np.ndarray:
        """FP16 bits of C[ms[i], ns[i]] for one group."""
        A, SFA, B, SFB = _u8(A), _u8(SFA), _u8(B), _u8(SFB)
        ms = np.ascontiguousarray(ms, dtype=np.int32)
        ns = np.ascontiguousarray(ns, dtype=np.int32)
        out = np.zeros(ms.shape[0], dtype=np.uint16)
        rc = self.L.nvfp4_oracle_gemm_elements(_p(A, _u8p), _p(SFA, _u8p), _p(B, _u8p),
                                               _p(SFB, _u8p), M, N, K, _p(ms, _i32p),
                                               _p(ns, _i32p), ms.shape[0], _p(out, _u16p))
        if rc != 0:
            raise ValueError("oracle gemm_elements failed")
        return out

    def gemm_fixed(self, A, SFA, B, SFB, M: int, N: int, K: int) -> np.ndarray:
        """Exact int64 sums in units of 2^-20 (independent accumulation)."""
        A, SFA, B, SFB = _u8(A), _u8(SFA), _u8(B), _u8(SFB)
        out = np.zeros((M, N), dtype=np.int64)
        rc = self.L.nvfp4_oracle_gemm_fixed(_p(A, _u8p), _p(SFA, _u8p), _p(B, _u8p),
                                            _p(SFB, _u8p), _p(out, _i64p), M, N, K)
        if rc != 0:
            raise ValueError("oracle gemm_fixed failed")
        return out

    def group_gemm(self, groups, threads: int = 0):
        """groups: objects with A, SFA, B, SFB (row-major scales), M, N, K.
        Returns a list of uint16 [M, N] arrays of FP16 bits."""
        return [self.gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, threads=threads)
                for g in groups]

    # fused epilogue -------------------------------------------------------------
    def bf16_rne_bits(self, x: float) -> int:
        return int(self.L.nvfp4_oracle_bf16_rne(float(x)))

    def silu(self, x: float) -> float:
        return float(self.L.nvfp4_oracle_silu(float(x)))

    def epilogue(self, acc, alpha: float = 1.0, swiglu: bool = False, bf16: bool = False):
        """From the exact float64 sums acc [M, N] of one group: alpha * acc,
        or the SwiGLU of 128-row gate / up blocks ([M, N/2]); FP16 or BF16
        bits (uint16)."""
        acc = np.ascontiguousarray(acc, dtype=np.float64)
        M, N = acc.shape
        out = np.zeros((M, N // 2 if swiglu else N), dtype=np.uint16)
        if M and self.L.nvfp4_oracle_epilogue(_p(acc, _f64p), M, N, float(alpha), int(swiglu),
                                              int(bf16), _p(out, _u16p)) != 0:
            raise ValueError("oracle epilogue failed")
        return out

    def gemm_ex(self, A, SFA, B, SFB, M, N, K, alpha=1.0, swiglu=False, bf16=False, threads=0):
        """One group through the fused epilogue."""
        _, acc = self.gemm(A, SFA, B, SFB, M, N, K, threads=threads, want_acc=True)
        return self.epilogue(acc, alpha, swiglu, bf16)

    # quantisation ---------------------------------------------------------------
    def e4m3_rne(self, v: float) -> int:
        return int(self.L.nvfp4_oracle_e4m3_rne(float(v)))

    def e2m1_rne(self, q: float) -> int:
        return int(self.L.nvfp4_oracle_e2m1_rne(float(q)))

    def quantize(self, x_bits, rows: int, K: int, bf16: bool = False):
        """x_bits: uint16 [rows, K] FP16 (or BF16) bits.  Returns (codes
        uint8 [rows, K/2], row-major E4M3FN scales uint8 [rows, K/16])."""
        x = np.ascontiguousarray(np.asarray(x_bits, dtype=np.uint16))
        assert x.size == rows * K
        codes = np.zeros((rows, K // 2), dtype=np.uint8)
        sf = np.zeros((rows, K // 16), dtype=np.uint8)
        if rows and self.L.nvfp4_oracle_quantize(_p(x, _u16p), 1 if bf16 else 0, rows, K,
                                                 _p(codes, _u8p), _p(sf, _u8p)) != 0:
            raise ValueError("oracle quantize failed")
        return codes, sf

    # scale-factor layout ------------------------------------------------------
    def sf_tiled_bytes(self, rows: int, K: int) -> int:
        return int(self.L.nvfp4_oracle_sf_tiled_bytes(rows, K))

    def sf_relayout(self, src, rows: int, K: int) -> np.ndarray:
        src = _u8(src)
        assert src.size == rows * K // 16
        dst = np.full(self.sf_tiled_bytes(rows, K), 0xAB, dtype=np.uint8)
        if dst.size and self.L.nvfp4_oracle_sf_relayout(_p(src, _u8p), _p(dst, _u8p),
                                                         rows, K) != 0:
            raise ValueError("oracle relayout failed")
        return dst

    def sf_unrelayout(self, tiled, rows: int, K: int) -> np.ndarray:
        tiled = _u8(tiled)
        dst = np.zeros((rows, K // 16), dtype=np.uint8)
        if rows and self.L.nvfp4_oracle_sf_unrelayout(_p(tiled, _u8p), _p(dst, _u8p),
                                                       rows, K) != 0:
            raise ValueError("oracle unrelayout failed")
        return dst


_default = None


def get() -> Oracle:
    """The oracle built from oracle/nvfp4_oracle.c."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
