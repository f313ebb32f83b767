"""GPU parity of the reverse mode (``kda_recurrent_bwd``) against the fp64
oracle backward, which tests/test_oracle_backward.py pins to central finite
differences of the forward oracle.

Both sides take the same inputs (bf16 inputs are rounded once and read as
exact values by the oracle), so the comparison measures the fp32 arithmetic
of the kernel.  Tolerance: relative L2 <= 1e-4 on each gradient, the fp32
bound the forward path meets; tensors whose reference is all zero must come
out zero."""
import numpy as np
import pytest
import torch

import linear_attention_layer_gb300 as kda
import oracle
import workloads
from tests.parity import as64, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = 1e-4
NAMES = ("dq", "dk", "dv", "dz", "dbeta", "d_initial")


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.load()
    torch.cuda.set_device(0)


def _cotangents(p, seed, with_final=True):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    T, H, _ = p.q.shape
    dv = p.v.shape[-1]
    N = len(p.cu_seqlens_host) - 1
    d_out = torch.randn((T, H, dv), device=DEV, generator=g).to(p.q.dtype)
    d_fin = (torch.randn((N, H, p.q.shape[-1], dv), device=DEV, generator=g)
             if with_final else None)
    return d_out, d_fin


def _compare(got, ref, tol=TOL):
    errs = {}
    for name, x, r in zip(NAMES, got, ref):
        r = as64(r)
        if not np.any(r):
            assert not np.any(as64(x)), f"{name}: expected zeros"
            errs[name] = 0.0
            continue
        errs[name] = rel_l2(x, r)
    bad = {k: v for k, v in errs.items() if v > tol}
    assert not bad, f"rel-L2 above {tol}: {bad} (all: {errs})"
    return errs


def _run(p, d_out, d_fin, a_log=None):
    grads = kda.recurrent_bwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state, d_out,
                              d_fin, cu_seqlens_host=p.cu_seqlens_host, a_log=a_log)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return grads


# lengths around the 8-token state spacing and the 64-token staging blocks
RAGGED = [1, 7, 8, 9, 0, 63, 64, 65, 130]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_backward_small_ragged(dtype):
    p = workloads.random_problem(RAGGED, 2, 128, 128, dtype, z_std=1.5, init_std=0.1, seed=21,
                                 device=DEV)
    d_out, d_fin = _cotangents(p, 3)
    got = _run(p, d_out, d_fin)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin)
    _compare(got, ref)


def test_backward_gate_log_scale():
    p = workloads.random_problem([100, 33], 3, 128, 128, torch.bfloat16, z_std=1.0,
                                 init_std=0.2, seed=22, device=DEV)
    a_log = torch.tensor([0.7, -1.2, 0.0], dtype=torch.float32, device=DEV)
    d_out, d_fin = _cotangents(p, 4)
    got = _run(p, d_out, d_fin, a_log=a_log)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin, a_log=a_log.cpu().numpy())
    _compare(got, ref)


def test_backward_no_initial_state_no_final_gradient():
    p = workloads.random_problem([70, 5], 2, 128, 128, torch.float32, seed=23, device=DEV)
    d_out, _ = _cotangents(p, 5, with_final=False)
    got = _run(p, d_out, None)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, None, d_out, None)
    _compare(got, ref)


def test_backward_only_final_gradient():
    """d out = 0: the gradient flows from the final state alone (and a
    zero-length sequence hands it straight to its initial state)."""
    p = workloads.random_problem([40, 0, 17], 1, 128, 128, torch.bfloat16, init_std=0.3,
                                 seed=24, device=DEV)
    d_out, d_fin = _cotangents(p, 6)
    d_out.zero_()
    got = _run(p, d_out, d_fin)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin)
    _compare(got, ref)
    assert torch.equal(got[5][1], d_fin[1])


@pytest.mark.parametrize("z_mean", [-2.0, 6.0])
def test_backward_decay_extremes(z_mean):
    """Near-saturated gates (alpha near e^-5) and slow decay (alpha near 1)."""
    p = workloads.random_problem([300], 2, 128, 128, torch.bfloat16, z_mean=z_mean,
                                 init_std=0.5, seed=25, device=DEV)
    d_out, d_fin = _cotangents(p, 7)
    got = _run(p, d_out, d_fin)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin)
    _compare(got, ref)


def test_backward_prefill_workload_sampled():
    """The 4 x 4096-token, 16-head prefill workload in one launch; two
    (sequence, head) pairs recomputed by the oracle."""
    p = workloads.prefill_workload("prefill", device=DEV)
    d_out, d_fin = _cotangents(p, 8)
    got = _run(p, d_out, d_fin)
    cu = p.cu_seqlens_host
    for n, h in [(0, 0), (3, 11)]:
        a, b = cu[n], cu[n + 1]
        sl = lambda x: x[a:b, h:h + 1].cpu()
        ref = oracle.backward(sl(p.q), sl(p.k), sl(p.v), sl(p.z), sl(p.beta), [0, b - a], None,
                              sl(d_out), d_fin[n:n + 1, h:h + 1].cpu())
        mine = [g[a:b, h:h + 1] for g in got[:5]] + [got[5][n:n + 1, h:h + 1]]
        _compare(mine, ref)


def test_backward_all_sequences_empty():
    """No tokens at all: the only gradient is the final state's, handed to the
    initial state unchanged."""
    p = workloads.random_problem([0, 0], 2, 128, 128, torch.bfloat16, init_std=0.3, seed=26,
                                 device=DEV)
    d_out = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device=DEV)
    d_fin = torch.randn((2, 2, 128, 128), device=DEV)
    got = _run(p, d_out, d_fin)
    assert torch.equal(got[5], d_fin)
    assert all(g.numel() == 0 for g in got[:5])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_backward_gate_per_head(dtype):
    """One gate logit per (token, head) (the scalar-alpha case): z and dz are
    [T, H].  The oracle runs the per-channel gate with the logit broadcast over
    the key channels, so the head's dz is the sum of its channel terms."""
    p = workloads.random_problem(RAGGED, 3, 128, 128, dtype, z_std=1.5, init_std=0.1, seed=27,
                                 device=DEV)
    zh = p.z[:, :, 0].contiguous()
    A = torch.tensor([0.5, -0.4, 1.2])
    d_out, d_fin = _cotangents(p, 7)
    got = kda.recurrent_bwd(p.q, p.k, p.v, zh, p.beta, p.cu_seqlens, p.initial_state, d_out,
                            d_fin, cu_seqlens_host=p.cu_seqlens_host, a_log=A.to(DEV))
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert got[3].shape == zh.shape
    zb = zh.cpu()[:, :, None].expand(-1, -1, 128).contiguous()
    ref = list(oracle.backward(p.q, p.k, p.v, zb, p.beta, p.cu_seqlens_host, p.initial_state,
                               d_out, d_fin, a_log=A))
    ref[3] = ref[3].sum(axis=-1)
    _compare(got, ref)


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (64, 32)])
def test_backward_small_dims(dk, dv):
    """dk or dv below 128 (zero-padded to 128 channels around the kernel):
    every gradient against the oracle, with the gate log-scale, and with one
    gate per head."""
    p = workloads.random_problem(RAGGED, 2, dk, dv, torch.bfloat16, z_std=1.5, init_std=0.1,
                                 seed=40 + dk + dv, device=DEV)
    A = torch.tensor([0.4, -0.7])
    d_out, d_fin = _cotangents(p, 9)
    got = kda.recurrent_bwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state, d_out,
                            d_fin, cu_seqlens_host=p.cu_seqlens_host, a_log=A.to(DEV))
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin, a_log=A)
    _compare(got, ref)
    zh = p.z[:, :, 0].contiguous()
    got = kda.recurrent_bwd(p.q, p.k, p.v, zh, p.beta, p.cu_seqlens, None, d_out, None,
                            cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    zb = zh.cpu()[:, :, None].expand(-1, -1, dk).contiguous()
    ref = list(oracle.backward(p.q, p.k, p.v, zb, p.beta, p.cu_seqlens_host, None, d_out, None))
    ref[3] = ref[3].sum(axis=-1)
    _compare(got, ref)
