"""The N > 1 path of bench.py on CPU: two gloo ranks, each running its own
shard (seed = rank) with no data-path collective, a barrier around the timed
region, the max of the per-rank times, and whole-job throughput = all ranks'
tokens / that max.  The per-rank work here is the fp64 oracle on a tiny
workload (the GPU kernels need a GPU)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import oracle
    import workloads
    r, w, local = bench.dist_info()
    assert (r, w, local) == (rank, world, rank)
    d = bench.init_dist(w, "gloo")
    # each rank its own shard of the same shape, seeded by rank
    p = workloads.random_problem([40, 23], 2, 16, 16, torch.float32, init_std=0.1, seed=r)
    bench.barrier(d)
    out, fin, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state)
    my_time = 0.25 + 0.5 * r  # stand-in per-rank elapsed seconds
    bench.barrier(d)
    t_max = bench.max_over_ranks(my_time, d, "cpu")
    value = bench.weak_scaling_value(p.total_tokens, w, t_max)
    np.save(os.path.join(outdir, f"rank{r}.npy"),
            np.array([t_max, value, float(np.abs(out).sum())]))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_weak_scaling(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    assert r0[0] == r1[0] == 0.75           # both ranks see the max time
    assert r0[1] == r1[1] == pytest.approx(63 * 2 / 0.75 / 1e6)
    assert r0[2] != r1[2]                   # independent shards (different seeds)
