"""Pins for the CPU oracle, written as functions of an oracle instance.

``test_oracle_pins.py`` runs them against the oracle (all must pass);
``test_oracle_mutants.py`` runs them against copies of the oracle with one
plausible mistake planted each (at least one must fail).  Nothing here calls
the oracle's own decoders to produce an expected value: expected values come
from the golden fixtures (published format tables), from PyTorch's
float8_e4m3fn conversion, from numpy's float16 rounding, from closed forms and
from an independent dense float64 expansion.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --- independent decoders (published tables / library conversions) --------

def golden_e2m1() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                out[int(c, 16)] = float(v)
    return out


def golden_e4m3_points() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "e4m3fn_points.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                out[int(c, 16)] = float(v)
    return out


def golden_atom_offsets() -> list:
    out = []
    with open(os.path.join(GOLDEN, "sf_atom_offsets.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(tuple(int(x) for x in line.split()))
    return out


def torch_e4m3_table() -> np.ndarray:
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


E2M1_TABLE = None


def e2m1_table() -> np.ndarray:
    global E2M1_TABLE
    if E2M1_TABLE is None:
        g = golden_e2m1()
        E2M1_TABLE = np.array([g[c] for c in range(16)], dtype=np.float64)
    return E2M1_TABLE


def dense(codes: np.ndarray, sf: np.ndarray, K: int) -> np.ndarray:
    """Dense float64 [rows, K] expansion: low nibble of byte i is element 2i."""
    rows = codes.shape[0]
    lo = codes & 0x0F
    hi = codes >> 4
    elem = np.empty((rows, K), dtype=np.int64)
    elem[:, 0::2] = lo
    elem[:, 1::2] = hi
    vals = e2m1_table()[elem]
    scales = torch_e4m3_table()[sf.astype(np.int64)]
    return vals * np.repeat(scales, 16, axis=1)


def brute_force_fp16_bits(A, SFA, B, SFB, K) -> np.ndarray:
    Ad = dense(A, SFA, K)
    Bd = dense(B, SFB, K)
    ref = Ad @ Bd.T
    return ref.astype(np.float16).view(np.uint16)


# --- random inputs -----------------------------------------------------------

def rand_case(rng, M, N, K, full_scale_range=False):
    A = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    if full_scale_range:
        # every finite E4M3FN byte, either sign (the oracle must not care)
        pool = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=np.uint8)
        SFA = rng.choice(pool, size=(M, K // 16))
        SFB = rng.choice(pool, size=(N, K // 16))
    else:
        def sc(rows):
            e = rng.integers(-4, 1, size=(rows, K // 16))
            m = rng.integers(0, 8, size=(rows, K // 16))
            return (((e + 7) << 3) | m).astype(np.uint8)
        SFA, SFB = sc(M), sc(N)
    return A, SFA, B, SFB


# --- the checks --------------------------------------------------------------

def check_e2m1_table(o):
    g = golden_e2m1()
    for c in range(16):
        v = o.e2m1(c)
        assert v == g[c] and math.copysign(1, v) == math.copysign(1, g[c]), (c, v, g[c])


def check_e4m3_all_codes(o):
    t = torch_e4m3_table()
    for b in range(256):
        v = o.e4m3fn(b)
        if math.isnan(t[b]):
            assert math.isnan(v), b
        else:
            assert v == t[b], (hex(b), v, t[b])
    for b, v in golden_e4m3_points().items():
        got = o.e4m3fn(b)
        assert (math.isnan(v) and math.isnan(got)) or got == v, (hex(b), got, v)


def check_fp16_rounding(o, seed=5):
    rng = np.random.default_rng(seed)
    xs = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-9, 6, size=2000))
    # exact ties between neighbouring halves, both parities, normal and subnormal
    h = rng.integers(1, 0x7BFF, size=600).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    xs += list((lo + hi) / 2)
    xs += list(-(lo + hi) / 2)
    xs += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
           3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11,
           1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0, float("inf"), float("-inf")]
    for x in xs:
        with np.errstate(over="ignore"):
            want = int(np.array(x, dtype=np.float64).astype(np.float16).view(np.uint16))
        got = o.fp16_rne_bits(float(x))
        assert got == want, (x, hex(got), hex(want))
    assert o.fp16_rne_bits(float("nan")) & 0x7C00 == 0x7C00


def check_brute_force_tiny(o, seed=11):
    rng = np.random.default_rng(seed)
    for (M, N, K) in [(1, 1, 16), (3, 5, 16), (7, 2, 64), (8, 8, 256), (5, 3, 64), (2, 7, 256)]:
        A, SFA, B, SFB = rand_case(rng, M, N, K)
        got = o.gemm(A, SFA, B, SFB, M, N, K, threads=2)
        want = brute_force_fp16_bits(A, SFA, B, SFB, K)
        assert np.array_equal(got, want), (M, N, K)
        els = o.gemm_elements(A, SFA, B, SFB, M, N, K,
                              np.repeat(np.arange(M), N), np.tile(np.arange(N), M))
        assert np.array_equal(els.reshape(M, N), want), (M, N, K)


def check_brute_force_grouped(o, seed=12):
    """A grouped call (a list of groups) against per-group brute force."""
    rng = np.random.default_rng(seed)
    shapes = [(4, 6, 64), (1, 3, 256), (6, 1, 16)]
    cases = [rand_case(rng, *s) for s in shapes]
    for (M, N, K), (A, SFA, B, SFB) in zip(shapes, cases):
        got = o.gemm(A, SFA, B, SFB, M, N, K)
        assert np.array_equal(got, brute_force_fp16_bits(A, SFA, B, SFB, K))


def check_fixed_point(o, seed=13):
    rng = np.random.default_rng(seed)
    for (M, N, K, full) in [(6, 5, 256, True), (4, 9, 512, True), (3, 4, 2048, False),
                            (2, 3, 7168, False)]:
        A, SFA, B, SFB = rand_case(rng, M, N, K, full_scale_range=full)
        _, acc = o.gemm(A, SFA, B, SFB, M, N, K, want_acc=True)
        fx = o.gemm_fixed(A, SFA, B, SFB, M, N, K)
        assert np.all(np.abs(fx) < 2 ** 53)
        assert np.array_equal(acc * 2.0 ** 20, fx.astype(np.float64)), (M, N, K)


def check_single_nonzero(o, seed=14):
    rng = np.random.default_rng(seed)
    e2 = e2m1_table()
    e4 = torch_e4m3_table()
    M, N, K = 5, 7, 256
    for _ in range(12):
        A = np.zeros((M, K // 2), np.uint8)
        B = np.zeros((N, K // 2), np.uint8)
        m0, n0, k0 = int(rng.integers(M)), int(rng.integers(N)), int(rng.integers(K))
        ca, cb = int(rng.integers(1, 16)), int(rng.integers(1, 16))
        if ca == 8:
            ca = 9
        if cb == 8:
            cb = 10
        A[m0, k0 // 2] = ca << 4 if k0 % 2 else ca
        B[n0, k0 // 2] = cb << 4 if k0 % 2 else cb
        _, SFA, _, SFB = rand_case(rng, M, N, K)
        C = o.gemm(A, SFA, B, SFB, M, N, K).view(np.float16).astype(np.float64)
        want = np.zeros((M, N))
        want[m0, n0] = np.float16(e2[ca] * e4[SFA[m0, k0 // 16]] * e2[cb] * e4[SFB[n0, k0 // 16]])
        assert np.array_equal(C, want), (m0, n0, k0, ca, cb)


def check_all_ones_power_of_two(o):
    """Every code 1.0 (nibble 0x2) with sa * sb = 2^k gives C = K * 2^k
    exactly (+inf once that passes the largest finite FP16, 65504)."""
    for K in (256, 1024):
        M, N = 3, 4
        A = np.full((M, K // 2), 0x22, np.uint8)
        B = np.full((N, K // 2), 0x22, np.uint8)
        for ka in range(-4, 1):
            for kb in range(-4, 8):
                SFA = np.full((M, K // 16), (ka + 7) << 3, np.uint8)   # 2^ka exactly
                SFB = np.full((N, K // 16), (kb + 7) << 3, np.uint8)
                C = o.gemm(A, SFA, B, SFB, M, N, K).view(np.float16).astype(np.float64)
                want = K * 2.0 ** (ka + kb)
                if want > 65504.0:          # past the largest finite half
                    want = np.inf
                assert np.all(C == want), (K, ka, kb, C[0, 0])


def check_zero_scales(o, seed=15):
    rng = np.random.default_rng(seed)
    M, N, K = 4, 6, 512
    A, SFA, B, SFB = rand_case(rng, M, N, K)
    C = o.gemm(A, np.zeros_like(SFA), B, SFB, M, N, K)
    assert np.all(C.view(np.float16).astype(np.float64) == 0.0)
    C = o.gemm(A, SFA, B, np.zeros_like(SFB), M, N, K)
    assert np.all(C.view(np.float16).astype(np.float64) == 0.0)


def check_nibble_order(o):
    """A nonzero only at k=0 (low nibble of byte 0), B only at k=1 (high
    nibble): the product never meets, C = 0.  Both at k=1: C = a*b."""
    K, M, N = 256, 1, 1
    SF = np.full((1, K // 16), 0x38, np.uint8)       # 1.0
    A = np.zeros((1, K // 2), np.uint8)
    B = np.zeros((1, K // 2), np.uint8)
    A[0, 0] = 0x02           # element 0 = 1.0
    B[0, 0] = 0x40           # element 1 = 2.0
    C = o.gemm(A, SF, B, SF, M, N, K).view(np.float16).astype(np.float64)
    assert C[0, 0] == 0.0
    A[0, 0] = 0x50           # element 1 = 3.0
    C = o.gemm(A, SF, B, SF, M, N, K).view(np.float16).astype(np.float64)
    assert C[0, 0] == 6.0


def check_scale_blocks(o):
    """Ones everywhere, SFA distinct per 16-block, SFB = 1: each block
    contributes 16 * its own scale, so C = 16 * sum of the row's scales;
    row m and column n see only their own scales."""
    M, N, K = 3, 2, 512
    A = np.full((M, K // 2), 0x22, np.uint8)
    B = np.full((N, K // 2), 0x22, np.uint8)
    e4 = torch_e4m3_table()
    rng = np.random.default_rng(16)
    SFA = rng.integers(0x20, 0x48, size=(M, K // 16)).astype(np.uint8)
    SFB = np.full((N, K // 16), 0x38, np.uint8)
    SFB[1, :] = 0x40                                  # column 1 doubled
    C = o.gemm(A, SFA, B, SFB, M, N, K).view(np.float16).astype(np.float64)
    for m in range(M):
        s = 16.0 * e4[SFA[m]].sum()
        assert C[m, 0] == np.float16(s), (m, C[m, 0], s)
        assert C[m, 1] == np.float16(2 * s), (m, C[m, 1], 2 * s)


def check_signs(o):
    K = 256
    SF = np.full((1, K // 16), 0x38, np.uint8)
    A = np.zeros((1, K // 2), np.uint8)
    B = np.zeros((2, K // 2), np.uint8)
    A[0, 3] = 0x09           # element 6 = -0.5
    B[0, 3] = 0x02           # element 6 = 1.0
    B[1, 3] = 0x0C           # element 6 = -2.0
    SFB = np.full((2, K // 16), 0x38, np.uint8)
    C = o.gemm(A, SF, B, SFB, 1, 2, K).view(np.float16).astype(np.float64)
    assert C[0, 0] == -0.5 and C[0, 1] == 1.0, C


def check_row_and_column_split(o, seed=17):
    """Row m of C depends only on row m of A (and column n only on row n of
    B): splitting A or B and concatenating the outputs changes nothing; so
    does permuting the groups of a grouped call."""
    rng = np.random.default_rng(seed)
    M, N, K = 9, 11, 512
    A, SFA, B, SFB = rand_case(rng, M, N, K)
    full = o.gemm(A, SFA, B, SFB, M, N, K)
    top = o.gemm(A[:4], SFA[:4], B, SFB, 4, N, K)
    bot = o.gemm(A[4:], SFA[4:], B, SFB, M - 4, N, K)
    assert np.array_equal(np.vstack([top, bot]), full)
    left = o.gemm(A, SFA, B[:6], SFB[:6], M, 6, K)
    right = o.gemm(A, SFA, B[6:], SFB[6:], M, N - 6, K)
    assert np.array_equal(np.hstack([left, right]), full)
    # a row-range call equals the corresponding rows of the full call
    part = o.gemm(A, SFA, B, SFB, M, N, K, rows=(2, 7))
    assert np.array_equal(part[2:7], full[2:7]) and not part[:2].any() and not part[7:].any()
    # so does a call for a list of rows, in any order
    pick = [8, 0, 5, 5, 3]
    assert np.array_equal(o.gemm_rows(A, SFA, B, SFB, M, N, K, pick), full[pick])


def check_transpose_symmetry(o, seed=18):
    """Swapping the operands transposes C (the sum is symmetric in A, B)."""
    rng = np.random.default_rng(seed)
    M, N, K = 5, 8, 256
    A, SFA, B, SFB = rand_case(rng, M, N, K)
    c1 = o.gemm(A, SFA, B, SFB, M, N, K)
    c2 = o.gemm(B, SFB, A, SFA, N, M, K)
    assert np.array_equal(c1, c2.T)


def check_relayout(o, seed=19):
    rng = np.random.default_rng(seed)
    for rows, K in [(1, 64), (128, 256), (200, 512), (300, 1024), (256, 7168)]:
        src = rng.integers(0, 256, size=(rows, K // 16), dtype=np.uint8)
        t = o.sf_relayout(src, rows, K)
        assert t.size == ((rows + 127) // 128) * (K // 64) * 512
        assert np.array_equal(o.sf_unrelayout(t, rows, K), src)
        # a permutation plus zero padding: byte histogram preserved
        pad = t.size - src.size
        hs = np.bincount(src.ravel(), minlength=256)
        hs[0] += pad
        assert np.array_equal(np.bincount(t, minlength=256), hs)
    for rows, K, r, j, off in golden_atom_offsets():
        src = np.zeros((rows, K // 16), np.uint8)
        src[r, j] = 0x5A
        t = o.sf_relayout(src, rows, K)
        nz = np.flatnonzero(t)
        assert nz.tolist() == [off], (rows, K, r, j, nz[:4], off)


# --- NVFP4 quantisation --------------------------------------------------

def _f32(v):
    return float(np.float32(v))


def check_quant_e4m3_vs_torch(o, seed=21):
    """The scale rounding against PyTorch's float8_e4m3fn conversion (round
    to nearest even) on random in-range values and on every exact midpoint
    between neighbouring E4M3FN values; above 448 the oracle saturates."""
    rng = np.random.default_rng(seed)
    vals = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(440.0), size=2000)).astype(np.float32)
    pts = sorted(golden_e4m3_points().items())
    pos = sorted(v for _, v in pts if 0 < v < float("inf") and v == v)
    grid = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, np.array(pos, dtype=np.float32)])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([o.e4m3_rne(float(v)) for v in vals], dtype=np.uint8)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(ref[i])) for i in bad[:5]]
    for v in (448.0, 449.0, 464.0, 1e6, 5e37, 3.4e38):
        assert o.e4m3_rne(v) == 0x7E, v
    assert o.e4m3_rne(0.0) == 0 and o.e4m3_rne(-3.0) == 0


# q -> E2M1 code, from the grid {0, .5, 1, 1.5, 2, 3, 4, 6} written out by
# hand: nearest value, ties to the even code, 6 above, zero without sign
_E2M1_CASES = [
    (0.0, 0x0), (0.24, 0x0), (0.25, 0x0), (0.26, 0x1), (0.5, 0x1), (0.74, 0x1), (0.75, 0x2),
    (1.25, 0x2), (1.26, 0x3), (1.75, 0x4), (2.49, 0x4), (2.5, 0x4), (2.51, 0x5), (3.49, 0x5),
    (3.5, 0x6), (4.99, 0x6), (5.0, 0x6), (5.01, 0x7), (6.0, 0x7), (100.0, 0x7),
    (-0.1, 0x0), (-0.25, 0x0), (-0.3, 0x9), (-1.75, 0xC), (-6.5, 0xF), (-3.0, 0xD),
    (1e30, 0x7), (-1e30, 0xF), (6.7e35, 0x7),
]


def check_quant_e2m1_rounding(o):
    for q, code in _E2M1_CASES:
        got = o.e2m1_rne(q)
        assert got == code, (q, got, code)


def _half_bits(vals):
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


def check_quant_blocks(o):
    """Hand-made blocks: exact scale 1 (absmax 6), an all-zero block, a block
    whose scale rounds to zero, a saturating block, a negative absmax, and the
    nibble order; FP16 and BF16 inputs of the same values agree."""
    K = 64
    x = np.zeros((2, K), dtype=np.float32)
    x[0, 0:16] = [6, -6, 3, 1.5, 0.5, -0.25, 0.75, 2, 0, 1, -1, 4, 5, 2.5, -3.5, 0.1]
    # block 1 of row 0 stays zero
    x[0, 32:48] = 0.005                     # absmax / 6 < 2^-10: scale 0
    x[0, 48:64] = [60000] + [1000] * 15     # scale saturates at 448
    x[1, 0:16] = [-12] + [1] * 15           # negative absmax: scale 2
    x[1, 16:32] = np.arange(16)            # scale 15/6 = 2.5
    for bf16 in (False, True):
        if bf16:
            bits = (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
        else:
            bits = _half_bits(x)
        codes, sf = o.quantize(bits, 2, K, bf16=bf16)
        assert sf[0].tolist() == [0x38, 0x00, 0x00, 0x7E], sf[0]
        assert sf[1, 0] == 0x40 and sf[1, 1] == 0x42, sf[1]     # 2.0, 2.5
        lo = codes[0, :8] & 0xF
        hi = codes[0, :8] >> 4
        first = np.empty(16, dtype=np.uint8)
        first[0::2], first[1::2] = lo, hi
        # 6,-6,3,1.5,.5,-.25,.75,2,0,1,-1,4,5,2.5,-3.5,.1 -> codes
        assert first.tolist() == [0x7, 0xF, 0x5, 0x3, 0x1, 0x0, 0x2, 0x4,
                                  0x0, 0x2, 0xA, 0x6, 0x6, 0x4, 0xE, 0x0], first
        assert not codes[0, 8:24].any()                 # zero block and scale-0 block
        assert (codes[0, 24] & 0xF) == 0x7 and (codes[0, 24] >> 4) == 0x4   # 60000/448 -> 6, 1000/448 = 2.23 -> 2
        # row 1 block 0: -12/2 = -6 -> 0xF, 1/2 = .5 -> 0x1
        assert codes[1, 0] == (0xF | (0x1 << 4))
        # row 1 block 1: i / 2.5 for i = 0..15
        exp = [o.e2m1_rne(np.float32(i) / np.float32(2.5)) for i in range(16)]
        got = [(codes[1, 8 + i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
        assert got == exp, (got, exp)


def check_quant_vs_float64_generator(o, seed=23):
    """Against the workloads' own per-block quantiser (float64 decisions,
    written independently): on Gaussian FP16 inputs every scale and all but
    rare rounding-boundary codes agree, and no code is off by more than one
    grid step."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from block_scaled_nvfp4_group_gb300 import workloads
    rng = np.random.default_rng(seed)
    rows, K = 64, 1024
    x16 = rng.standard_normal((rows, K)).astype(np.float16)
    codes, sf = o.quantize(x16.view(np.uint16), rows, K)
    c64, s64 = workloads.quantize_nvfp4(x16.astype(np.float64))
    assert (sf == s64).mean() > 0.999, (sf != s64).sum()
    same = sf == s64
    a = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(rows, K)
    b = np.stack([c64 & 0xF, c64 >> 4], axis=-1).reshape(rows, K)
    blockok = np.repeat(same, 16, axis=1)
    diff = (a != b) & blockok
    assert diff.mean() < 1e-3, diff.sum()
    mag = lambda c: c & 7
    assert (np.abs(mag(a[diff]).astype(int) - mag(b[diff]).astype(int)) <= 1).all()


# --- fused epilogue (per-tensor scale, BF16 output, SwiGLU) --------------

def check_bf16_rounding(o, seed=31):
    """Against PyTorch's float32 -> bfloat16 conversion (round to nearest
    even) on float32 values: normals over the whole range, subnormals, exact
    ties, overflow."""
    rng = np.random.default_rng(seed)
    vals = np.concatenate([
        rng.standard_normal(3000) * np.exp(rng.uniform(-80, 80, 3000)),
        rng.standard_normal(500) * 1e-39,
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3.3895e38, 3.39e38, 0.0]),
    ]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([o.bf16_rne_bits(float(v)) for v in vals], dtype=np.uint16)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def check_silu(o, seed=32):
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.standard_normal(200) * 20, [0.0, -800.0, 800.0]])
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    got = np.array([o.silu(float(v)) for v in x])
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-300), np.abs(got - ref).max()


def check_epilogue_mapping(o):
    """SwiGLU pairs output column 128 j + c with gate column 256 j + c and up
    column 256 j + 128 + c; alpha scales both before the SiLU; the plain
    epilogue scales every sum."""
    M, N = 3, 512
    acc = np.zeros((M, N))
    acc[1, 256 + 5] = 2.0
    acc[1, 256 + 128 + 5] = 3.0
    acc[2, 7] = -4.0
    acc[2, 128 + 7] = 0.5
    alpha = 0.75
    out = o.epilogue(acc, alpha=alpha, swiglu=True)
    assert out.shape == (M, N // 2)
    silu = lambda v: float(torch.nn.functional.silu(torch.tensor(v, dtype=torch.float64)))
    exp = np.zeros((M, N // 2), dtype=np.float16)
    exp[1, 128 + 5] = silu(alpha * 2.0) * alpha * 3.0
    exp[2, 7] = silu(alpha * -4.0) * alpha * 0.5
    assert np.array_equal(out.view(np.float16), exp), np.argwhere(out.view(np.float16) != exp)
    out_b = o.epilogue(acc, alpha=alpha, swiglu=True, bf16=True)
    exp_b = torch.from_numpy(exp.astype(np.float32)).to(torch.bfloat16)
    got_b = torch.from_numpy(out_b.view(np.int16)).view(torch.bfloat16)
    assert (got_b.float() - exp_b.float()).abs().max() <= 2 ** -7 * exp_b.float().abs().max()
    plain = o.epilogue(acc, alpha=alpha).view(np.float16)
    assert plain.shape == (M, N) and plain[1, 261] == np.float16(1.5) and plain[2, 135] == np.float16(0.375)
    assert np.count_nonzero(plain) == 4


# --- quantisation decisions, exhaustive over the 16-bit input formats ---

# the E2M1 magnitude grid's rounding boundaries (midpoints of neighbours) and
# whether a value exactly on one goes up: ties go to the even code, i.e. up
# at .75, 1.75 and 3.5, down at .25, 1.25, 2.5 and 5
_E2M1_MIDS = [(0.25, False), (0.75, True), (1.25, False), (1.75, True), (2.5, False), (3.5, True),
              (5.0, False)]


def _finite_16bit(bf16: bool):
    """(bits, float64 values) of every finite FP16 or BF16 number"""
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        if bf16:
            vals = (bits << 16).view(np.float32).astype(np.float64)
        else:
            vals = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    keep = np.isfinite(vals)
    return bits[keep].astype(np.uint16), vals[keep]


def _to_bits(v: np.ndarray, bf16: bool) -> np.ndarray:
    if bf16:
        return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return v.astype(np.float16).view(np.uint16)


def _e2m1_by_thresholds(x: np.ndarray, s: float) -> np.ndarray:
    a = np.abs(x)
    mag = np.zeros(x.shape, dtype=np.uint8)
    for mid, tie_up in _E2M1_MIDS:
        t = mid * s                      # <= 6 significant bits: exact in float64
        mag += (a >= t) if tie_up else (a > t)
    return np.where((x < 0) & (mag != 0), mag | 8, mag).astype(np.uint8)


def check_quant_codes_exhaustive(o):
    """Every finite FP16 and BF16 value x against every positive E4M3FN scale
    s it can meet (|x| <= 6 s, in blocks whose absmax 6 s fixes the scale at
    s): the oracle's code of x / s must be the rounding onto the magnitude
    grid written as exact float64 comparisons of |x| with the grid's
    midpoints times s.  With 11 or 8 significant bits, x / s is never within
    half a single-precision ulp of a midpoint unless it is one, so taking the
    quotient in single precision first changes no code; a single-precision
    x * (1/s) does (it moves exact ties)."""
    grid = torch_e4m3_table()
    for bf16 in (False, True):
        bits, vals = _finite_16bit(bf16)
        for c in range(1, 0x7F):
            s = float(grid[c])
            xs = vals[np.abs(vals) <= 6.0 * s]
            nblk = -(-xs.size // 15)
            blocks = np.zeros((nblk, 16), dtype=np.float64)
            blocks[:, 0] = 6.0 * s                               # absmax / 6 = s exactly
            body = np.zeros(nblk * 15, dtype=np.float64)
            body[:xs.size] = xs
            blocks[:, 1:] = body.reshape(nblk, 15)
            rows = -(-nblk // 64)
            x = np.zeros((rows * 64, 16), dtype=np.float64)
            x[:nblk] = blocks
            codes, sf = o.quantize(_to_bits(x.reshape(rows, 64 * 16), bf16), rows, 64 * 16, bf16=bf16)
            assert (sf.reshape(-1)[:nblk] == c).all(), ("scale", bf16, c)
            got = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(rows * 64, 16)[:nblk]
            want = _e2m1_by_thresholds(blocks, s)
            bad = np.argwhere(got != want)
            assert bad.size == 0, [("bf16" if bf16 else "fp16", s, float(blocks[i, j]), int(got[i, j]),
                                    int(want[i, j])) for i, j in bad[:4]]


def check_quant_scales_exhaustive(o):
    """Every finite FP16 and BF16 value as a block's absmax: the oracle's scale
    must be E4M3FN(absmax / 6) written as exact float64 comparisons of absmax
    with six times the midpoints of neighbouring E4M3FN values (ties to the
    even code, 448 for anything above it, 0 for zero)."""
    grid = torch_e4m3_table()[:0x7F].astype(np.float64)    # codes 0..126, increasing
    mids6 = 6.0 * (grid[1:] + grid[:-1]) / 2.0             # exact: few significant bits
    for bf16 in (False, True):
        bits, vals = _finite_16bit(bf16)
        amax = np.abs(vals)
        code = np.searchsorted(mids6, amax, side="left")    # midpoints strictly below amax
        tie = np.isin(amax, mids6)
        # on a midpoint between codes k and k+1 (code == k here): the even one
        k = code[tie]
        code[tie] = np.where(k % 2 == 0, k, k + 1)
        code = np.minimum(code, 0x7E)
        K = 1024
        n = amax.size
        rows = -(-n // (K // 16))
        x = np.zeros(rows * (K // 16) * 16, dtype=np.float64)
        x[0:n * 16:16] = vals
        _, sf = o.quantize(_to_bits(x.reshape(rows, K), bf16), rows, K, bf16=bf16)
        got = sf.reshape(-1)[:n]
        bad = np.flatnonzero(got != code)
        assert bad.size == 0, [(float(vals[i]), int(got[i]), int(code[i])) for i in bad[:4]]


ALL_CHECKS = [
    check_e2m1_table, check_e4m3_all_codes, check_fp16_rounding, check_brute_force_tiny,
    check_brute_force_grouped, check_fixed_point, check_single_nonzero,
    check_all_ones_power_of_two, check_zero_scales, check_nibble_order, check_scale_blocks,
    check_signs, check_row_and_column_split, check_transpose_symmetry, check_relayout,
    check_quant_e4m3_vs_torch, check_quant_e2m1_rounding, check_quant_blocks,
    check_quant_vs_float64_generator, check_bf16_rounding, check_silu, check_epilogue_mapping,
    check_quant_codes_exhaustive, check_quant_scales_exhaustive,
]
