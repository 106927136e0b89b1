"""The N > 1 host path on CPU with two gloo ranks: expert-parallel sharding
covers every group exactly once and the per-rank results (computed here by
the oracle) concatenate to the single-process result; the max-over-ranks
timing reduction; per-rank seeds."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from block_scaled_nvfp4_group_gb300 import shard


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from block_scaled_nvfp4_group_gb300 import workloads
        from oracle import oracle
        shapes = [(40, 64, 256), (0, 64, 256), (130, 32, 512), (7, 128, 256), (64, 64, 768)]
        groups = workloads.make_groups(shapes, seed=77)
        mine = shard.shard_groups(shapes, world, rank)
        res = {}
        for i in mine:
            g = groups[i]
            if g.M:
                res[i] = oracle.get().gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, threads=1)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), idx=np.array(mine),
                 **{f"c{i}": v for i, v in res.items()})
        m = shard.max_over_ranks(float(rank * 10 + 3))
        with open(os.path.join(out_dir, f"max{rank}.txt"), "w") as f:
            f.write(str(m))
    finally:
        dist.destroy_process_group()


def test_two_rank_shard_and_max(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    from block_scaled_nvfp4_group_gb300 import workloads
    from oracle import oracle
    shapes = [(40, 64, 256), (0, 64, 256), (130, 32, 512), (7, 128, 256), (64, 64, 768)]
    groups = workloads.make_groups(shapes, seed=77)
    seen = []
    for r in range(2):
        d = np.load(tmp_path / f"rank{r}.npz")
        seen += d["idx"].tolist()
        for i in d["idx"].tolist():
            g = groups[i]
            if g.M:
                want = oracle.get().gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, threads=1)
                assert np.array_equal(d[f"c{i}"], want)
        assert float(open(tmp_path / f"max{r}.txt").read()) == 13.0
    assert sorted(seen) == list(range(len(shapes)))


def test_shard_balance_and_edges():
    shapes = [(366, 4096, 7168), (261, 4096, 7168), (336, 4096, 7168), (45, 4096, 7168),
              (223, 4096, 7168), (107, 4096, 7168), (317, 4096, 7168), (349, 4096, 7168)]
    for world in (1, 2, 3, 4, 8):
        parts = [shard.shard_groups(shapes, world, r) for r in range(world)]
        assert sorted(sum(parts, [])) == list(range(8))
        loads = [sum(shapes[i][0] for i in p) for p in parts]
        assert max(loads) - min(loads) <= max(s[0] for s in shapes)
    with pytest.raises(ValueError):
        shard.shard_groups(shapes, 2, 2)
    assert shard.rank_seed(1001, 0) == 1001 and shard.rank_seed(1001, 3) == 4001
    assert shard.max_over_ranks(2.5) == 2.5
