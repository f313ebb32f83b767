"""Context parallelism: one batch of long sequences cut along the token axis
across the ranks of a process group, one rank per GPU.

The scheme is the one the pages describe for KDA across devices
(blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "第二层"): the
state update is affine in the state, so rank r first folds its own shard of
every sequence into an affine summary S_out = M_r S_in + S~_r
(``kda_chunk_fwd_summary``); one all-gather exchanges the summaries (M: dk x dk,
S~: dk x dv fp32 per sequence and head -- 128 KiB per head at dk = dv = 128);
a prefix scan over the summaries of ranks 0 .. r-1 (``kda_state_scan``) gives
the state entering rank r's shard; and an ordinary prefill of the shard from
that state (``kda_chunk_fwd``) writes its outputs.  Rank R-1's final states
are the sequences' final states.

Layout: every rank holds, for each of the same N sequences, one contiguous
piece (possibly empty); rank r's piece of a sequence directly follows rank
r-1's.  Each rank passes its own packed pieces and their cu_seqlens (device
and host copies), and the same ``initial_state`` (the states before rank 0's
pieces) or None.

The collective is torch.distributed's all_gather on the given group (NCCL for
GPU tensors).  The three compute steps are the library's, through ``ops``;
the default ``LibraryOps`` calls libkda and fails loudly if it is missing.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import chunk_fwd, chunk_fwd_summary, state_scan


class LibraryOps:
    """The three per-rank compute steps, on the GPU through libkda."""

    def summary(self, q, k, v, z, beta, cu_seqlens, cu_seqlens_host, a_log=None):
        return chunk_fwd_summary(q, k, v, z, beta, cu_seqlens, cu_seqlens_host,
                                 workspace="auto", a_log=a_log)

    def scan(self, transitions, offsets, initial_state, count):
        return state_scan(transitions, offsets, initial_state, count=count)

    def prefill(self, q, k, v, z, beta, cu_seqlens, cu_seqlens_host, initial_state, a_log=None):
        return chunk_fwd(q, k, v, z, beta, cu_seqlens, initial_state,
                         cu_seqlens_host=cu_seqlens_host, workspace="auto", a_log=a_log)


def chunk_fwd_context_parallel(q, k, v, z, beta, cu_seqlens, cu_seqlens_host,
                               initial_state=None, *, group=None, a_log=None, ops=None,
                               broadcast_final_state=False):
    """This rank's part of a context-parallel prefill (see the module text).

    q, k, v, z, beta, cu_seqlens, cu_seqlens_host: this rank's pieces of the
    N sequences, packed as for ``chunk_fwd``; initial_state: [N, H, dk, dv]
    fp32, the same on every rank, or None.  Returns (out, final_state): this
    rank's outputs and the states after its pieces -- on the last rank the
    sequences' final states (on every rank with ``broadcast_final_state``).
    """
    ops = LibraryOps() if ops is None else ops
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    m, s = ops.summary(q, k, v, z, beta, cu_seqlens, cu_seqlens_host, a_log)
    ms = [torch.empty_like(m) for _ in range(world)]
    ss = [torch.empty_like(s) for _ in range(world)]
    dist.all_gather(ms, m.contiguous(), group=group)
    dist.all_gather(ss, s.contiguous(), group=group)
    entry = ops.scan(torch.stack(ms), torch.stack(ss), initial_state, rank)
    out, fin = ops.prefill(q, k, v, z, beta, cu_seqlens, cu_seqlens_host, entry, a_log)
    if broadcast_final_state:
        dist.broadcast(fin, src=dist.get_global_rank(group, world - 1) if group else world - 1,
                       group=group)
    return out, fin


def shard_bounds(cu_seqlens_host, world):
    """A balanced cut of each sequence into ``world`` consecutive pieces:
    for sequence n, rank r takes tokens [b[n][r], b[n][r+1]) (positions
    within the sequence).  Pieces end on multiples of 64 tokens where
    possible, so that every rank's chunks line up with the whole sequence's."""
    out = []
    for n in range(len(cu_seqlens_host) - 1):
        length = int(cu_seqlens_host[n + 1]) - int(cu_seqlens_host[n])
        chunks = (length + 63) // 64
        b = [min(length, 64 * ((chunks * r) // world)) for r in range(world)] + [length]
        out.append(b)
    return out
