"""Context parallelism across two gloo ranks on the CPU.

Each rank holds its piece of every sequence and runs the library's
context-parallel driver (linear_attention_layer_gb300.context_parallel):
affine summary of its pieces, all-gather of the summaries over the process
group, prefix scan to its entering states, prefill of its pieces.  The
compute steps here are the fp64 oracle's (the GPU kernels need a GPU; the
single-GPU test of the same steps on the kernels is
tests/test_gpu_context_parallel.py), so this checks the exchange and the
ordering of the scheme: the ranks' outputs put together must equal one
oracle pass over the whole sequences, and the last rank's final states the
sequences' final states."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LENGTHS = [300, 40, 0, 129]
H, DK, DV = 2, 16, 8


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The driver's three compute steps, on the CPU oracle (test stand-in)."""

    def __init__(self, oracle):
        self.oracle = oracle

    def summary(self, q, k, v, z, beta, cu_seqlens, cu_seqlens_host, a_log=None):
        m, s = self.oracle.affine_summary(q, k, v, z, beta, cu_seqlens_host, a_log=a_log)
        return torch.from_numpy(m), torch.from_numpy(s)

    def scan(self, transitions, offsets, initial_state, count):
        return torch.from_numpy(self.oracle.state_scan(transitions, offsets, initial_state,
                                                       count=count))

    def prefill(self, q, k, v, z, beta, cu_seqlens, cu_seqlens_host, initial_state, a_log=None):
        out, fin, _ = self.oracle.recurrent(q, k, v, z, beta, cu_seqlens_host, initial_state,
                                            a_log=a_log)
        return torch.from_numpy(out), torch.from_numpy(fin)


def _problem():
    import workloads
    return workloads.random_problem(LENGTHS, H, DK, DV, torch.float32, init_std=0.3, seed=7)


def _pieces(p, bounds, r):
    """Rank r's packed pieces: (token index list, local cu_seqlens)."""
    idx, cu = [], [0]
    for n, b in enumerate(bounds):
        start = p.cu_seqlens_host[n]
        idx += list(range(start + b[r], start + b[r + 1]))
        cu.append(cu[-1] + b[r + 1] - b[r])
    return idx, cu


def _worker(rank, world, port, outdir):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from linear_attention_layer_gb300 import context_parallel as cp
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    p = _problem()
    bounds = cp.shard_bounds(p.cu_seqlens_host, world)
    idx, cu = _pieces(p, bounds, rank)
    sel = lambda x: x[idx].contiguous()
    a_log = torch.tensor([0.4, -0.7])
    out, fin = cp.chunk_fwd_context_parallel(
        sel(p.q), sel(p.k), sel(p.v), sel(p.z), sel(p.beta),
        torch.tensor(cu, dtype=torch.int32), cu, p.initial_state, a_log=a_log,
        ops=OracleOps(oracle), broadcast_final_state=True)
    np.save(os.path.join(outdir, f"out{rank}.npy"), out.numpy())
    np.save(os.path.join(outdir, f"fin{rank}.npy"), fin.numpy())
    np.save(os.path.join(outdir, f"idx{rank}.npy"), np.array(idx, dtype=np.int64))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_context_parallel_equals_one_pass(tmp_path):
    import oracle
    from linear_attention_layer_gb300 import context_parallel as cp
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    p = _problem()
    ref_out, ref_fin, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host,
                                           p.initial_state, a_log=torch.tensor([0.4, -0.7]))
    out = np.full_like(ref_out, np.nan)
    for r in range(world):
        idx = np.load(tmp_path / f"idx{r}.npy")
        out[idx] = np.load(tmp_path / f"out{r}.npy")
        # broadcast_final_state: every rank holds the sequences' final states
        np.testing.assert_allclose(np.load(tmp_path / f"fin{r}.npy"), ref_fin, rtol=0,
                                   atol=1e-11)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-11)
    # both ranks had work, and one piece was empty (the 40-token sequence's first)
    bounds = cp.shard_bounds(p.cu_seqlens_host, world)
    assert bounds[0] == [0, 128, 300] and bounds[1] == [0, 0, 40]


def test_shard_bounds_cover_each_sequence_in_order():
    from linear_attention_layer_gb300 import context_parallel as cp
    cu = [0, 1000, 1000, 1064, 1065]
    for world in (1, 2, 3, 8):
        for n, b in enumerate(cp.shard_bounds(cu, world)):
            L = cu[n + 1] - cu[n]
            assert len(b) == world + 1 and b[0] == 0 and b[-1] == L
            assert all(x <= y for x, y in zip(b, b[1:]))
            assert all(x % 64 == 0 for x in b[:-1])
