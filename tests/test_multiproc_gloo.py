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


def _ep_worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from block_scaled_nvfp4_group_gb300 import workloads
        from oracle import oracle
        idx, groups = workloads.expert_parallel_groups("tiny", world, rank)
        res = {f"c{gi}": oracle.get().gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, threads=1)
               for gi, g in zip(idx, groups)}
        flops = sum(2 * g.M * g.N * g.K for g in groups)
        np.savez(os.path.join(out_dir, f"ep{rank}.npz"), idx=np.array(idx), flops=flops, **res)
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_split(tmp_path):
    """The split bench.py uses under torchrun: two ranks share one grouped
    call of two copies of the workload's groups; every group is computed by
    exactly one rank, each rank holds the same FLOPs, copy 0 is the workload
    itself and copy 1 has its own data."""
    port = _free_port()
    mp.spawn(_ep_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    from block_scaled_nvfp4_group_gb300 import workloads
    from oracle import oracle
    shapes = workloads.expert_parallel_shapes("tiny", 2)
    assert shapes == [(64, 256, 256), (128, 256, 256)] * 2
    base = workloads.make_workload("tiny").groups
    seen, flops, outs = [], [], {}
    for r in range(2):
        d = np.load(tmp_path / f"ep{r}.npz")
        seen += d["idx"].tolist()
        flops.append(int(d["flops"]))
        for gi in d["idx"].tolist():
            outs[gi] = d[f"c{gi}"]
    assert sorted(seen) == [0, 1, 2, 3]
    assert flops[0] == flops[1]
    for i, g in enumerate(base):
        ref = oracle.get().gemm(g.A, g.SFA, g.B, g.SFB, g.M, g.N, g.K, threads=1)
        assert np.array_equal(outs[i], ref)
    # copy 1 draws its own inputs: same shapes, different C
    assert outs[2].shape == outs[0].shape and not np.array_equal(outs[2], outs[0])
    # one rank alone gets the workload itself
    idx1, g1 = workloads.expert_parallel_groups("tiny", 1, 0)
    assert idx1 == [0, 1] and all(np.array_equal(a.A, b.A) for a, b in zip(g1, base))
