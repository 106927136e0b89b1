"""Helpers shared by the GPU tests: device problems, oracle comparison."""
from __future__ import annotations

import numpy as np
import pytest
import torch

RTOL = 1e-3     # |C - C_oracle| <= RTOL * |C_oracle| + ATOL, elementwise
ATOL = 1e-2


def require_gb300():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cc = torch.cuda.get_device_capability(0)
    if cc != (10, 3):
        pytest.skip(f"needs compute capability 10.3, found {cc}")


def compare_fp16(got_bits: np.ndarray, ref_bits: np.ndarray, what: str) -> None:
    """Elementwise |gpu - oracle| <= 1e-3 |oracle| + 1e-2, and the same
    non-finite values where the oracle has them."""
    g = got_bits.view(np.float16).astype(np.float64)
    r = ref_bits.view(np.float16).astype(np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: non-finite pattern differs"
    assert np.array_equal(g[~fin], r[~fin]), f"{what}: inf/nan values differ"
    err = np.abs(g[fin] - r[fin])
    bad = err > RTOL * np.abs(r[fin]) + ATOL
    if bad.any():
        idx = np.argwhere(fin)[np.flatnonzero(bad)[:5]]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"first at {idx.tolist()}: gpu {g[tuple(idx[0])]} "
                             f"oracle {r[tuple(idx[0])]}")


BF16_RTOL = 2.0 ** -7   # one BF16 ulp: the FP32 sum may round to the neighbour of the exact sum's BF16


def compare_bf16(got_bits: np.ndarray, ref_bits: np.ndarray, what: str) -> None:
    """Elementwise |gpu - oracle| <= 2^-7 |oracle| + 1e-2 on BF16 outputs."""
    g = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (ref_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    fin = np.isfinite(r)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: non-finite pattern differs"
    err = np.abs(g[fin] - r[fin])
    bad = err > BF16_RTOL * np.abs(r[fin]) + ATOL
    if bad.any():
        idx = np.argwhere(fin)[np.flatnonzero(bad)[:5]]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first at "
                             f"{idx.tolist()}: gpu {g[tuple(idx[0])]} oracle {r[tuple(idx[0])]}")


KINDS = {"stream": 0, "wide": 1, "compute": 2, "wide512": 3, "wide_p2": 4, "wide_p4": 5,
         "pair": 6, "wide_sk": 7, "swap": 8}


class gemm_env:
    """Force the GEMM configuration (and optionally the L2 prefetch distance)
    through the library's environment knobs, restoring them afterwards."""

    def __init__(self, kind=None, pf=None):
        import os
        self.os = os
        self.vals = {"NVFP4_GEMM_KIND": None if kind is None else str(KINDS[kind]),
                     "NVFP4_PF_STAGES": None if pf is None else str(pf)}
        self.saved = {}

    def __enter__(self):
        for k, v in self.vals.items():
            self.saved[k] = self.os.environ.get(k)
            if v is None:
                self.os.environ.pop(k, None)
            else:
                self.os.environ[k] = v
        return self

    def __exit__(self, *exc):
        for k, v in self.saved.items():
            if v is None:
                self.os.environ.pop(k, None)
            else:
                self.os.environ[k] = v
