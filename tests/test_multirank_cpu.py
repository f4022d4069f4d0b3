"""The multi-rank host logic of the benchmark on CPU (gloo, world size 2):
each rank owns independent sessions (seeded by rank), and the reported
numbers are the max step time and the summed bytes over ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from bit_kv_cache_nvfp4_gb300 import workloads as wl
    w = wl.make_workload("tiny", seed=rank)
    t_ms = 1.0 + rank                      # rank 1 is slower
    nbytes = 1000.0 * (rank + 1)
    max_ms, tot = bench.reduce_over_ranks(t_ms, nbytes)
    world_env, rank_env, local_env = bench.dist_env()
    out[rank] = torch.tensor([max_ms, tot, float(w.topk.sum()), float(rank_env), float(world_env)])
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    out = torch.zeros(world, 5).share_memory_()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert torch.all(out[:, 0] == 2.0)            # max over ranks
    assert torch.all(out[:, 1] == 3000.0)         # sum over ranks
    assert out[0, 2] != out[1, 2]                 # independent session sets per rank
    assert out[0, 3] == 0 and out[1, 3] == 1 and torch.all(out[:, 4] == 2)


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.5, 10) == (3.5, 10.0)
