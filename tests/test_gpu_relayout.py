"""Scale-factor relayout kernel against the oracle's permutation
(byte-exact), including ragged row counts and the zero padding."""
import numpy as np
import pytest
import torch

from gpu_util import require_gb300
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gb300()


@pytest.mark.parametrize("rows,K", [(1, 256), (127, 256), (128, 512), (129, 768), (200, 1024),
                                    (300, 7168), (4096, 7168), (400, 2048), (7168, 2048),
                                    (1000, 4096)])
def test_relayout_matches_oracle(rows, K):
    from block_scaled_nvfp4_group_gb300 import ops
    rng = np.random.default_rng(rows * 7 + K)
    src = rng.integers(0, 256, size=(rows, K // 16), dtype=np.uint8)
    want = oracle.get().sf_relayout(src, rows, K)
    d_src = torch.from_numpy(src).cuda().reshape(-1)
    out = torch.full((ops.sf_tiled_bytes(rows, K),), 0xCD, dtype=torch.uint8, device="cuda")
    ops.sf_relayout(d_src, rows, K, out=out)
    got = out.cpu().numpy()
    assert np.array_equal(got, want)


def test_grouped_relayout_one_launch():
    from block_scaled_nvfp4_group_gb300 import ops
    rng = np.random.default_rng(3)
    shapes = [(64, 256), (1, 512), (333, 2048), (128, 7168), (0, 256), (4096, 256)]
    items, wants = [], []
    for rows, K in shapes:
        src = rng.integers(0, 256, size=(rows, K // 16), dtype=np.uint8)
        d_src = torch.from_numpy(src).cuda().reshape(-1) if rows else torch.empty(0, dtype=torch.uint8, device="cuda")
        dst = torch.full((max(ops.sf_tiled_bytes(rows, K), 16),), 0xCD, dtype=torch.uint8, device="cuda")
        items.append((d_src, dst, rows, K))
        wants.append(oracle.get().sf_relayout(src, rows, K) if rows else None)
    ops.sf_relayout_group(items)
    torch.cuda.synchronize()
    for (d_src, dst, rows, K), want in zip(items, wants):
        if rows:
            assert np.array_equal(dst.cpu().numpy()[:want.size], want), (rows, K)
        else:
            assert (dst.cpu().numpy() == 0xCD).all()


def test_relayout_many_descriptors_split_launches():
    from block_scaled_nvfp4_group_gb300 import ops
    rng = np.random.default_rng(5)
    items, wants = [], []
    for i in range(70):                       # more than one launch's worth
        rows, K = int(rng.integers(1, 300)), 256 * int(rng.integers(1, 4))
        src = rng.integers(0, 256, size=(rows, K // 16), dtype=np.uint8)
        dst = torch.empty(ops.sf_tiled_bytes(rows, K), dtype=torch.uint8, device="cuda")
        items.append((torch.from_numpy(src).cuda().reshape(-1), dst, rows, K))
        wants.append(oracle.get().sf_relayout(src, rows, K))
    ops.sf_relayout_group(items)
    for (_, dst, _, _), want in zip(items, wants):
        assert np.array_equal(dst.cpu().numpy(), want)
