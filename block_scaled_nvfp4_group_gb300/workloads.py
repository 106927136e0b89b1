"""Seeded synthetic inputs for the NVFP4 grouped GEMM.

This module only draws random bytes (and, for the quantised workload, rounds
Gaussian samples onto the E2M1 / E4M3FN grids).  It holds none of the GEMM's
arithmetic and serves the oracle side and the CUDA side alike.

Workloads (one list of groups each; every group holds A [M, K/2] and
B [N, K/2] as packed E2M1 codes, element 2i in the low nibble of byte i,
and plain row-major E4M3FN scales SFA [M, K/16], SFB [N, K/16]):

* ``tiny``      2 groups, N=K=256, M={64, 128}; uniform codes, scales
                2^e (1 + m/8) with e in [-4, 0], m in [0, 7].
* ``moe_gate_up`` 8 groups, N=4096, K=7168, M_g ~ U{40..400}; same draws.
* ``moe_down``  8 groups, N=7168, K=2048, M_g ~ U{40..400}; same draws.
* ``quantized`` 2 groups, M=512, N=3072, K=4096; N(0, 1) values quantised
                per 16-block (absmax / 6 rounded to E4M3FN, values rounded
                to the E2M1 grid, saturating at +-6).
* ``square``    4 groups, M=N=K=4096; uniform codes and scales.

The seed of workload i (in the order above) is 1000 + i.  Codes are uniform
over all 16 nibbles (each byte is two independent uniform nibbles).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

WORKLOADS = ("tiny", "moe_gate_up", "moe_down", "quantized", "square")


@dataclass
class Group:
    M: int
    N: int
    K: int
    A: np.ndarray      # uint8 [M, K/2]
    SFA: np.ndarray    # uint8 [M, K/16], row-major
    B: np.ndarray      # uint8 [N, K/2]
    SFB: np.ndarray    # uint8 [N, K/16], row-major


@dataclass
class Workload:
    name: str
    seed: int
    groups: list = field(default_factory=list)

    @property
    def flops(self) -> int:
        return sum(2 * g.M * g.N * g.K for g in self.groups)

    @property
    def algorithmic_bytes(self) -> int:
        """Unpadded bytes of A, B, SFA, SFB read and C written."""
        return sum(g.M * g.K // 2 + g.N * g.K // 2 + g.M * g.K // 16 + g.N * g.K // 16
                   + g.M * g.N * 2 for g in self.groups)

    @property
    def sf_bytes(self) -> int:
        return sum(g.M * g.K // 16 + g.N * g.K // 16 for g in self.groups)

    def shapes(self):
        return [(g.M, g.N, g.K) for g in self.groups]


def _uniform_codes(rng: np.random.Generator, rows: int, K: int) -> np.ndarray:
    return rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)


def _uniform_scales(rng: np.random.Generator, rows: int, K: int) -> np.ndarray:
    e = rng.integers(-4, 1, size=(rows, K // 16))
    m = rng.integers(0, 8, size=(rows, K // 16))
    return (((e + 7) << 3) | m).astype(np.uint8)


# --- quantisation used only by the ``quantized`` workload -----------------

_E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _round_to_e2m1_code(q: np.ndarray) -> np.ndarray:
    """Magnitude code (0..7) of |q| rounded to {0,.5,1,1.5,2,3,4,6}, ties to
    the even code, saturating at 6; the sign goes to bit 3."""
    a = np.minimum(np.abs(q), 6.0)
    code = np.searchsorted(_E2M1_MIDPOINTS, a, side="left")   # ties round down
    tie = np.isin(a, _E2M1_MIDPOINTS)
    code = np.where(tie & (code % 2 == 1), code + 1, code)    # ...then to even
    sign = (q < 0) & (code > 0)
    return (code | (sign.astype(np.int64) << 3)).astype(np.uint8)


def _round_to_e4m3(v: np.ndarray):
    """Non-negative v rounded to E4M3FN with ties to even, saturating at 448.
    Returns (code, rounded value)."""
    v = np.asarray(v, dtype=np.float64)
    out_val = np.zeros_like(v)
    out_code = np.zeros(v.shape, dtype=np.uint8)
    nz = v > 0
    x = np.minimum(v[nz], 448.0)
    _, ex = np.frexp(x)                       # x = f * 2^ex, f in [0.5, 1)
    qexp = np.maximum(ex - 4, -9)             # 4 significant bits; 2^-9 below 2^-6
    r = np.ldexp(x, -qexp)
    n = np.round(r)                           # numpy rounds half to even
    w = np.ldexp(n, qexp)
    w = np.minimum(w, 448.0)
    f2, e2 = np.frexp(w)
    sub = w < 2.0 ** -6
    mant_sub = np.ldexp(w, 9).astype(np.int64)
    efield = (e2 + 6).astype(np.int64)       # w = (2 f2) 2^(e2-1); bias 7
    mant = ((f2 * 2.0 - 1.0) * 8.0).astype(np.int64)
    code = np.where(sub, mant_sub, (efield << 3) | mant)
    out_val[nz] = w
    out_code[nz] = code.astype(np.uint8)
    return out_code, out_val


def quantize_nvfp4(x: np.ndarray):
    """Per-16-block NVFP4 quantisation of a float matrix [rows, K]:
    returns (packed codes [rows, K/2], scales [rows, K/16])."""
    rows, K = x.shape
    blocks = x.reshape(rows, K // 16, 16).astype(np.float64)
    absmax = np.abs(blocks).max(axis=2)
    sf_code, sf_val = _round_to_e4m3(absmax / 6.0)
    safe = np.where(sf_val > 0, sf_val, 1.0)
    q = np.where(sf_val[..., None] > 0, blocks / safe[..., None], 0.0)
    codes = _round_to_e2m1_code(q).reshape(rows, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return np.ascontiguousarray(packed), np.ascontiguousarray(sf_code)


# --- workload builders ------------------------------------------------------

def _uniform_group(rng, M, N, K) -> Group:
    A = _uniform_codes(rng, M, K)
    SFA = _uniform_scales(rng, M, K)
    B = _uniform_codes(rng, N, K)
    SFB = _uniform_scales(rng, N, K)
    return Group(M, N, K, A, SFA, B, SFB)


def make_groups(shapes, seed: int, kind: str = "uniform") -> list:
    """Groups of the given (M, N, K) shapes, drawn in order from one seed."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for (M, N, K) in shapes:
        if kind == "uniform":
            out.append(_uniform_group(rng, M, N, K))
        elif kind == "gaussian":
            A, SFA = quantize_nvfp4(rng.standard_normal((M, K)))
            B, SFB = quantize_nvfp4(rng.standard_normal((N, K)))
            out.append(Group(M, N, K, A, SFA, B, SFB))
        else:
            raise ValueError(kind)
    return out


def moe_m_sizes(seed: int, n_groups: int = 8, lo: int = 40, hi: int = 400):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(v) for v in rng.integers(lo, hi + 1, size=n_groups)]


def make_workload(name: str) -> Workload:
    idx = WORKLOADS.index(name)
    seed = 1000 + idx
    if name == "tiny":
        shapes = [(64, 256, 256), (128, 256, 256)]
        kind = "uniform"
    elif name == "moe_gate_up":
        shapes = [(m, 4096, 7168) for m in moe_m_sizes(seed)]
        kind = "uniform"
    elif name == "moe_down":
        shapes = [(m, 7168, 2048) for m in moe_m_sizes(seed)]
        kind = "uniform"
    elif name == "quantized":
        shapes = [(512, 3072, 4096)] * 2
        kind = "gaussian"
    elif name == "square":
        shapes = [(4096, 4096, 4096)] * 4
        kind = "uniform"
    else:
        raise ValueError(name)
    # the M draws use their own generator; the data generator is offset so
    # the two streams never overlap
    return Workload(name, seed, make_groups(shapes, seed + 7919, kind))


def describe(name: str) -> dict:
    """Shapes without generating data."""
    idx = WORKLOADS.index(name)
    seed = 1000 + idx
    if name == "tiny":
        shapes = [(64, 256, 256), (128, 256, 256)]
    elif name == "moe_gate_up":
        shapes = [(m, 4096, 7168) for m in moe_m_sizes(seed)]
    elif name == "moe_down":
        shapes = [(m, 7168, 2048) for m in moe_m_sizes(seed)]
    elif name == "quantized":
        shapes = [(512, 3072, 4096)] * 2
    else:
        shapes = [(4096, 4096, 4096)] * 4
    return {"name": name, "seed": seed, "shapes": shapes}


# --- expert-parallel batches (one process per GPU) --------------------------

def expert_parallel_shapes(name: str, world_size: int):
    """Shapes of the global grouped call that `world_size` ranks share: the
    workload's group list repeated `world_size` times (copy c holds the
    experts of rank c's worth of work), so each rank keeps about one
    workload's FLOPs (weak scaling)."""
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    return list(describe(name)["shapes"]) * world_size


def expert_parallel_groups(name: str, world_size: int, rank: int):
    """The groups of the global grouped call (expert_parallel_shapes) that
    `rank` owns, as (global indices, groups).  The split is
    shard.shard_groups (longest processing time first by FLOPs); copy 0 of
    the group list holds the workload's own data, copy c >= 1 draws group i
    from its own seed, so every rank can build exactly its groups.  With
    world_size 1 this is the workload itself."""
    from . import shard
    base = describe(name)
    n = len(base["shapes"])
    shapes = expert_parallel_shapes(name, world_size)
    mine = shard.shard_groups(shapes, world_size, rank)
    kind = "gaussian" if name == "quantized" else "uniform"
    own = None
    out = []
    for gi in mine:
        c, i = divmod(gi, n)
        if c == 0:
            if own is None:
                own = make_workload(name).groups
            out.append(own[i])
        else:
            seed = base["seed"] + 7919 + 1000 * c + i
            out.append(make_groups([shapes[gi]], seed, kind)[0])
    return mine, out
