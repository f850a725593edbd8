"""Host logic of the multi-rank benchmark path, run as two gloo ranks on the CPU:
each rank draws its own shard (distinct seeds, same shapes) and the timing is
the max over ranks; the data path itself has no collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from causal_gqa_attention_xt_gb300.inputs import WORKLOADS, make_inputs
    r, w, _ = bench.dist_env()
    wl = WORKLOADS["gqa_bf16"].with_(B=1, S=32)
    x = make_inputs(wl.with_(seed=bench.shard_seed(wl.seed, r)))
    mx = bench.reduce_max([float(r + 1), 10.0 - r, 0.5 * r])
    sums = torch.tensor([float(x["q"].float().sum())])
    gathered = [torch.zeros(1) for _ in range(w)]
    dist.all_gather(gathered, sums)
    out[rank] = (mx, [float(g) for g in gathered], tuple(x["q"].shape))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_take_max():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        mx, sums, shape = out[r]
        assert mx == [2.0, 10.0, 0.5]
        assert shape == (1, 32, 8, 64)
        assert sums[0] != sums[1]          # distinct shards
    assert out[0][1] == out[1][1]


def test_reduce_max_without_process_group_is_identity():
    import bench
    assert bench.reduce_max([1.0, 2.0]) == [1.0, 2.0]
