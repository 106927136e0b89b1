"""NVFP4 quantisation kernel against the CPU oracle, byte for byte (codes,
row-major scales and the tiled scale layout), and the quantise -> grouped
GEMM path against the oracle GEMM of the oracle's own quantisation."""
import numpy as np
import pytest
import torch

from gpu_util import compare_fp16, require_gb300
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gb300()


def _bits(x: np.ndarray, bf16: bool) -> np.ndarray:
    if bf16:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(x, dtype=np.float16).view(np.uint16)


def _run(x_bits: np.ndarray, bf16: bool):
    from block_scaled_nvfp4_group_gb300 import ops
    rows, K = x_bits.shape
    xt = torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16 if bf16 else torch.float16)
    codes, tiled, rm = ops.quantize(xt, want_rowmajor=True)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), tiled.cpu().numpy(), rm.cpu().numpy()


def _check(x: np.ndarray, bf16: bool, what: str):
    o = oracle.get()
    bits = _bits(x, bf16)
    rows, K = bits.shape
    codes, tiled, rm = _run(bits, bf16)
    rc, rs = o.quantize(bits, rows, K, bf16=bf16)
    bad = np.argwhere(codes != rc)
    assert bad.size == 0, f"{what}: {len(bad)} code bytes differ, first {bad[:3].tolist()}"
    assert np.array_equal(rm, rs), f"{what}: row-major scales differ"
    assert np.array_equal(tiled[:o.sf_tiled_bytes(rows, K)], o.sf_relayout(rs, rows, K)), \
        f"{what}: tiled scales differ"


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("rows,K", [(1, 64), (77, 128), (128, 256), (300, 1024), (513, 192)])
def test_gaussian(rows, K, bf16):
    rng = np.random.default_rng(rows * 7 + K)
    x = rng.standard_normal((rows, K)) * np.exp(rng.uniform(-3, 3, size=(rows, 1)))
    _check(x, bf16, f"gaussian {rows}x{K}")


@pytest.mark.parametrize("bf16", [False, True])
def test_edge_values(bf16):
    """All-zero blocks, blocks whose scale rounds to 0, saturating blocks,
    exact E2M1 ties (power-of-two scales), negative values that round to
    zero, subnormal FP16 inputs, and the largest finite FP16 / BF16."""
    K = 256
    rows = 8
    x = np.zeros((rows, K), dtype=np.float64)
    x[1, :] = 0.004                                      # scale 0
    x[2, :] = 60000.0 if not bf16 else 3e38              # saturation
    x[2, 1::2] = -1000.0
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -2.5, -5.0,
                     0.0, 1.0, -6.0, 4.0])
    x[3, :] = np.tile(ties, K // 16)                     # absmax 6: scale 1 exactly
    x[4, :] = np.tile(ties * 0.125, K // 16)             # scale 2^-3 exactly
    x[5, :] = np.tile([6.0] + [-0.01] * 15, K // 16)     # negatives rounding to zero
    x[6, :] = 2.0 ** -20                                 # FP16 subnormals
    x[6, ::16] = 2.0 ** -14
    x[7, :] = np.linspace(-65504, 65504, K) if not bf16 else np.linspace(-1e30, 1e30, K)
    _check(x, bf16, "edge values")


def test_workload_operands_full_size():
    """The quantized configuration's operands at full size (A 512 x 4096,
    B 3072 x 4096, Gaussian FP16), every byte."""
    rng = np.random.default_rng(2024)
    for rows in (512, 3072):
        _check(rng.standard_normal((rows, 4096)), False, f"operand {rows}x4096")


def test_quantize_then_gemm():
    """Quantise A and B on the GPU, run the grouped GEMM on the result, and
    compare with the oracle GEMM on the oracle's quantisation of the same
    inputs (the codes must already agree byte for byte)."""
    from block_scaled_nvfp4_group_gb300 import ops
    o = oracle.get()
    rng = np.random.default_rng(77)
    shapes = [(200, 512, 1024), (64, 256, 512)]
    items, refs = [], []
    for (M, N, K) in shapes:
        a = rng.standard_normal((M, K)).astype(np.float16)
        b = rng.standard_normal((N, K)).astype(np.float16)
        ca, ta, _ = ops.quantize(torch.from_numpy(a).cuda())
        cb, tb, _ = ops.quantize(torch.from_numpy(b).cuda())
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        items.append((ca, cb, ta, tb, C, M, N, K))
        ra, sa = o.quantize(a.view(np.uint16), M, K)
        rb, sb = o.quantize(b.view(np.uint16), N, K)
        refs.append(o.gemm(ra, sa, rb, sb, M, N, K))
    ops.group_gemm(items)
    torch.cuda.synchronize()
    for (M, N, K), it, ref in zip(shapes, items, refs):
        got = it[4].view(torch.int16).cpu().numpy().view(np.uint16)
        compare_fp16(got, ref, f"quantise->gemm {M}x{N}x{K}")


def test_rejects_bad_shapes():
    from block_scaled_nvfp4_group_gb300 import _abi
    lib = _abi.load()
    x = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    c = torch.zeros(4 * 32, dtype=torch.uint8, device="cuda")
    s = torch.zeros(512, dtype=torch.uint8, device="cuda")
    assert lib.nvfp4_quantize(x.data_ptr(), 0, 4, 48, c.data_ptr(), s.data_ptr(), None, None) == \
        _abi.NVFP4_ERR_INVALID_ARGUMENT
    assert lib.nvfp4_quantize(x.data_ptr() + 2, 0, 4, 64, c.data_ptr(), s.data_ptr(), None, None) == \
        _abi.NVFP4_ERR_MISALIGNED
    assert lib.nvfp4_quantize(x.data_ptr(), 0, 0, 64, c.data_ptr(), s.data_ptr(), None, None) == \
        _abi.NVFP4_OK


def _exhaustive_blocks(bf16: bool) -> np.ndarray:
    """16-element blocks that hit every positive E4M3FN scale s: each block is
    [6 s, x_1 .. x_15] with the x_i running through every finite FP16 (or
    BF16) magnitude in [0, 6 s], alternately negated, so every code and tie
    of every scale is formed (absmax 6 s gives exactly the scale s)."""
    o = oracle.get()
    dec = [o.e4m3fn(c) for c in range(128)]
    if bf16:
        mags = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        mags = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    blocks = []
    for code in range(1, 127):
        s = dec[code]
        a = 6.0 * s
        xs = mags[mags <= a]
        xs = np.where(np.arange(xs.size) % 2 == 1, -xs, xs)
        pad = (-xs.size) % 15
        xs = np.concatenate([xs, np.zeros(pad)]).reshape(-1, 15)
        blocks.append(np.concatenate([np.full((xs.shape[0], 1), a), xs], axis=1))
    return np.concatenate(blocks).reshape(-1)


@pytest.mark.parametrize("bf16", [False, True])
def test_exhaustive_values_and_scales(bf16):
    """Every finite FP16 / BF16 magnitude against every E4M3 scale it can
    meet, through the kernel, byte for byte against the oracle."""
    vals = _exhaustive_blocks(bf16)
    K = 4096
    vals = np.concatenate([vals, np.zeros((-vals.size) % K)])
    x = vals.reshape(-1, K)
    _check(x, bf16, f"exhaustive {'bf16' if bf16 else 'fp16'} {x.shape}")


@pytest.mark.parametrize("bf16", [False, True])
def test_every_absmax(bf16):
    """Every finite FP16 / BF16 magnitude as a block's absmax (blocks
    [a, -a/3, a/5, 0 ...]): the scale decision E4M3(absmax / 6) for every
    input value, and the codes of a few quotients per block, byte for byte
    against the oracle."""
    if bf16:
        a = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        a = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    blocks = np.zeros((a.size, 16))
    blocks[:, 0] = a
    blocks[:, 1] = -a / 3
    blocks[:, 2] = a / 5
    K = 4096
    vals = blocks.reshape(-1)
    vals = np.concatenate([vals, np.zeros((-vals.size) % K)])
    _check(vals.reshape(-1, K), bf16, f"every absmax {'bf16' if bf16 else 'fp16'}")
