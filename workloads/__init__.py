"""Seeded synthetic KDA inputs.

This module only draws random tensors with the shapes and distributions of
the five KDA workloads.  It holds none of the method's arithmetic and is the
one thing the oracle side (tests, CPU baseline) and the CUDA side (tests,
bench) share: both read the same materialised tensors.

Distributions: N(m, s) means mean m, standard deviation s.  q and k are
drawn N(0, 1) and divided by their Euclidean norm per (token, head) before
rounding to the io dtype (the workloads ask for L2-normalised q, k); v is
N(0, 1); z (gate logits, fp32) is N(z_mean, z_std); beta = 1 / (1 + e^-x)
with x ~ N(0, 1) (a write strength in (0, 1)); the optional initial state is
N(0, init_std) in fp32.  Draw order: q, k, v, z, x, state.  Sequence
lengths of the packed variable-length workload come from numpy's PCG64
seeded with `seed`, independent of the tensor draws.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass
class Problem:
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    z: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor  # int32 on the tensors' device
    cu_seqlens_host: list
    initial_state: Optional[torch.Tensor]
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self):
        return len(self.cu_seqlens_host) - 1

    @property
    def total_tokens(self):
        return self.cu_seqlens_host[-1]


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _unit_rows(x):
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)


def random_problem(lengths, num_heads, dk, dv, io_dtype=torch.bfloat16, *, z_mean=0.0,
                   z_std=1.0, init_std=None, seed=0, device="cpu", name="custom",
                   normalize_qk=True):
    """Packed variable-length batch with the module's distributions."""
    lengths = [int(x) for x in lengths]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T, H = int(cu[-1]), int(num_heads)
    g = _gen(device, seed)
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    q = torch.randn((T, H, dk), **f32)
    k = torch.randn((T, H, dk), **f32)
    if normalize_qk and T > 0:
        q, k = _unit_rows(q), _unit_rows(k)
    v = torch.randn((T, H, dv), **f32)
    z = torch.randn((T, H, dk), **f32) * z_std + z_mean
    beta = torch.sigmoid(torch.randn((T, H), **f32))
    s0 = None
    if init_std is not None:
        s0 = torch.randn((len(lengths), H, dk, dv), **f32) * init_std
    return Problem(
        name=name, q=q.to(io_dtype), k=k.to(io_dtype), v=v.to(io_dtype), z=z, beta=beta,
        cu_seqlens=torch.tensor(cu, dtype=torch.int32, device=device),
        cu_seqlens_host=[int(x) for x in cu], initial_state=s0,
        meta=dict(num_heads=H, dk=dk, dv=dv, dtype=str(io_dtype).replace("torch.", ""),
                  z_mean=z_mean, z_std=z_std, init_std=init_std, seed=seed))


def varlen_lengths(n=64, lo=256, hi=8192, seed=0):
    """Integer lengths uniform on [lo, hi] inclusive (numpy PCG64)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


# The five KDA workloads, by name.  Prefill ones return a Problem.
PREFILL_WORKLOADS = {
    "tiny": dict(lengths=[64], num_heads=1, dk=32, dv=32, io_dtype=torch.float32,
                 z_mean=0.0, z_std=1.0, init_std=None),
    "prefill": dict(lengths=[4096] * 4, num_heads=16, dk=128, dv=128,
                    io_dtype=torch.bfloat16, z_mean=0.0, z_std=1.5, init_std=None),
    "long": dict(lengths=[65536], num_heads=32, dk=128, dv=128, io_dtype=torch.bfloat16,
                 z_mean=2.0, z_std=1.0, init_std=None),
    # long-memory variant of "long" (parity only): alpha near e^-0.6
    "long_slow": dict(lengths=[65536], num_heads=32, dk=128, dv=128, io_dtype=torch.bfloat16,
                      z_mean=-2.0, z_std=1.0, init_std=None),
    "varlen": dict(lengths=None, num_heads=32, dk=128, dv=128, io_dtype=torch.bfloat16,
                   z_mean=0.0, z_std=1.0, init_std=0.1),
}

DESCRIPTIONS = {
    "tiny": "B=1 H=1 T=64 dk=dv=32 fp32, z~N(0,1), zero initial state",
    "prefill": "B=4 x T=4096 H=16 dk=dv=128 bf16, z~N(0,1.5), no initial state",
    "long": "B=1 T=65536 H=32 dk=dv=128 bf16, z~N(2,1), no initial state",
    "long_slow": "B=1 T=65536 H=32 dk=dv=128 bf16, z~N(-2,1), no initial state",
    "varlen": "64 seqs, lengths U{256..8192}, H=32 dk=dv=128 bf16, z~N(0,1), "
              "initial state N(0,0.1), final state returned",
    "decode": "256 requests x H=32, dk=dv=128, fp32 state N(0,0.1), bf16 q/k/v per step, "
              "z~N(0,1), 1000 steps",
}


def prefill_workload(name, device="cpu", seed=0):
    spec = dict(PREFILL_WORKLOADS[name])
    if spec["lengths"] is None:
        spec["lengths"] = varlen_lengths(seed=seed)
    return random_problem(seed=seed, device=device, name=name, **spec)


@dataclass
class DecodeProblem:
    state: torch.Tensor  # [N, H, dk, dv] fp32
    q: torch.Tensor      # [steps, N, H, dk]
    k: torch.Tensor
    v: torch.Tensor      # [steps, N, H, dv]
    z: torch.Tensor      # [steps, N, H, dk] fp32
    beta: torch.Tensor   # [steps, N, H] fp32
    meta: dict = field(default_factory=dict)


def decode_workload(num_requests=256, num_heads=32, dk=128, dv=128, steps=1000,
                    io_dtype=torch.bfloat16, state_std=0.1, seed=0, device="cpu"):
    """Batched decode: fresh per-step tokens for every live request."""
    g = _gen(device, seed)
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    N, H = num_requests, num_heads
    q = _unit_rows(torch.randn((steps, N, H, dk), **f32)).to(io_dtype)
    k = _unit_rows(torch.randn((steps, N, H, dk), **f32)).to(io_dtype)
    v = torch.randn((steps, N, H, dv), **f32).to(io_dtype)
    z = torch.randn((steps, N, H, dk), **f32)
    beta = torch.sigmoid(torch.randn((steps, N, H), **f32))
    state = torch.randn((N, H, dk, dv), **f32) * state_std
    return DecodeProblem(state=state, q=q, k=k, v=v, z=z, beta=beta,
                         meta=dict(num_requests=N, num_heads=H, dk=dk, dv=dv, steps=steps,
                                   seed=seed))
