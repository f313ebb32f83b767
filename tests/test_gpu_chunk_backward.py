"""GPU parity of the chunked tensor-core reverse mode (``kda_chunk_bwd``)
against the fp64 oracle backward, which tests/test_oracle_backward.py pins to
central finite differences of the forward oracle.

The chunk products run as bf16 tensor-core multiplies on operands split into
a high and a low bf16 part (16 significant bits, three multiplies per
product) with fp32 accumulation, and the log-decay gradient is summed without
cancelling terms, so the gradients carry fp32-class error.  Tolerance, per
gradient tensor: relative L2 <= 1e-4 (the fp32 bound kda_recurrent_bwd meets)
and max|err| <= 1e-2 RMS of the reference (the measured worst is about 1e-3
on the 4 x 4096 x 16 workload); tensors whose reference is all zero must come
out zero.  Each test prints the measured errors."""
import numpy as np
import pytest
import torch

import linear_attention_layer_gb300 as kda
import oracle
import workloads
from tests.parity import as64, max_over_rms, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL_REL = 1e-4
TOL_MAX = 1e-2
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


def _compare(got, ref, what=""):
    errs = {}
    for name, x, r in zip(NAMES, got, ref):
        r = as64(r)
        if not np.any(r):
            assert not np.any(as64(x)), f"{name}: expected zeros"
            errs[name] = (0.0, 0.0)
            continue
        errs[name] = (rel_l2(x, r), max_over_rms(x, r))
    print(f"{what}: " + ", ".join(f"{k} {a:.2e}/{m:.2e}" for k, (a, m) in errs.items()))
    bad = {k: v for k, v in errs.items() if v[0] > TOL_REL or v[1] > TOL_MAX}
    assert not bad, f"(rel-L2, max/RMS) above ({TOL_REL}, {TOL_MAX}): {bad}"
    return errs


def _run(p, d_out, d_fin, a_log=None, z=None):
    grads = kda.chunk_bwd(p.q, p.k, p.v, p.z if z is None else z, p.beta, p.cu_seqlens,
                          p.initial_state, d_out, d_fin, cu_seqlens_host=p.cu_seqlens_host,
                          a_log=a_log)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return grads


# lengths around the 16-token chunks and the 64-token state spacing
RAGGED = [1, 15, 16, 17, 0, 63, 64, 65, 130, 200]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_chunk_backward_small_ragged(dtype):
    p = workloads.random_problem(RAGGED, 2, 128, 128, dtype, z_std=1.5, init_std=0.1, seed=21,
                                 device=DEV)
    d_out, d_fin = _cotangents(p, 3)
    got = _run(p, d_out, d_fin)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin)
    _compare(got, ref, f"ragged {dtype}")


def test_chunk_backward_gate_log_scale():
    p = workloads.random_problem([100, 33], 3, 128, 128, torch.bfloat16, z_std=1.0,
                                 init_std=0.2, seed=22, device=DEV)
    a_log = torch.tensor([0.7, -1.2, 0.0], dtype=torch.float32, device=DEV)
    d_out, d_fin = _cotangents(p, 4)
    got = _run(p, d_out, d_fin, a_log=a_log)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin, a_log=a_log.cpu().numpy())
    _compare(got, ref, "gate log-scale")


def test_chunk_backward_no_initial_state_no_final_gradient():
    p = workloads.random_problem([70, 5], 2, 128, 128, torch.float32, seed=23, device=DEV)
    d_out, _ = _cotangents(p, 5, with_final=False)
    got = kda.chunk_bwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, None, d_out, None,
                        cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, None, d_out, None)
    _compare(got, ref, "no initial / final")


def test_chunk_backward_only_final_gradient():
    """d out = 0: the gradient flows from the final state alone (and a
    zero-length sequence hands it straight to its initial state)."""
    p = workloads.random_problem([40, 0, 17], 1, 128, 128, torch.bfloat16, init_std=0.3,
                                 seed=24, device=DEV)
    d_out, d_fin = _cotangents(p, 6)
    d_out.zero_()
    got = _run(p, d_out, d_fin)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin)
    _compare(got, ref, "final gradient only")
    assert torch.equal(got[5][1], d_fin[1])


@pytest.mark.parametrize("z_mean", [-2.0, 6.0])
def test_chunk_backward_decay_extremes(z_mean):
    """Near-saturated gates (alpha near e^-5: 16-token decay factors near
    e^-80) and slow decay (alpha near 1), over several 64-token blocks."""
    p = workloads.random_problem([300], 2, 128, 128, torch.bfloat16, z_mean=z_mean,
                                 init_std=0.5, seed=25, device=DEV)
    d_out, d_fin = _cotangents(p, 7)
    got = _run(p, d_out, d_fin)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin)
    _compare(got, ref, f"z mean {z_mean}")


def test_chunk_backward_long_sequence():
    """1,000 tokens (16 blocks of stored states, a ragged last chunk) next to
    short ones: the longest-first unit order and the block rebuild."""
    p = workloads.random_problem([1000, 37, 250], 2, 128, 128, torch.bfloat16, z_std=1.2,
                                 init_std=0.2, seed=28, device=DEV)
    d_out, d_fin = _cotangents(p, 11)
    got = _run(p, d_out, d_fin)
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin)
    _compare(got, ref, "long sequence")


def test_chunk_backward_all_sequences_empty():
    p = workloads.random_problem([0, 0], 2, 128, 128, torch.bfloat16, init_std=0.3, seed=26,
                                 device=DEV)
    d_out = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device=DEV)
    d_fin = torch.randn((2, 2, 128, 128), device=DEV)
    got = _run(p, d_out, d_fin)
    assert torch.equal(got[5], d_fin)
    assert all(g.numel() == 0 for g in got[:5])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_chunk_backward_gate_per_head(dtype):
    """One gate logit per (token, head): z and dz [T, H]; the oracle runs the
    per-channel gate with the logit broadcast, so dz is the channel sum."""
    p = workloads.random_problem(RAGGED, 3, 128, 128, dtype, z_std=1.5, init_std=0.1, seed=27,
                                 device=DEV)
    zh = p.z[:, :, 0].contiguous()
    A = torch.tensor([0.5, -0.4, 1.2])
    d_out, d_fin = _cotangents(p, 7)
    got = _run(p, d_out, d_fin, a_log=A.to(DEV), z=zh)
    assert got[3].shape == zh.shape
    zb = zh.cpu()[:, :, None].expand(-1, -1, 128).contiguous()
    ref = list(oracle.backward(p.q, p.k, p.v, zb, p.beta, p.cu_seqlens_host, p.initial_state,
                               d_out, d_fin, a_log=A))
    ref[3] = ref[3].sum(axis=-1)
    _compare(got, ref, f"per-head gate {dtype}")


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64)])
def test_chunk_backward_small_dims(dk, dv):
    """dk or dv below 128, zero-padded to 128 channels around the kernel."""
    p = workloads.random_problem(RAGGED, 2, dk, dv, torch.bfloat16, z_std=1.5, init_std=0.1,
                                 seed=40 + dk + dv, device=DEV)
    A = torch.tensor([0.4, -0.7])
    d_out, d_fin = _cotangents(p, 9)
    got = _run(p, d_out, d_fin, a_log=A.to(DEV))
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin, a_log=A)
    _compare(got, ref, f"dk {dk} dv {dv}")


def test_chunk_backward_matches_recurrent_on_prefill_workload():
    """The 4 x 4096-token, 16-head prefill workload in one launch: every
    gradient tensor against the per-token fp32 reverse mode on the GPU, and two
    (sequence, head) pairs against the oracle."""
    p = workloads.prefill_workload("prefill", device=DEV)
    d_out, d_fin = _cotangents(p, 8)
    got = _run(p, d_out, d_fin)
    ref = kda.recurrent_bwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state, d_out,
                            d_fin, cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    for name, x, r in zip(NAMES, got, ref):
        rel = float(torch.linalg.vector_norm((x - r).double()) /
                    torch.linalg.vector_norm(r.double()))
        rms = float(torch.sqrt(torch.mean(r.double() ** 2)))
        mx = float((x - r).abs().max()) / rms
        print(f"prefill workload vs recurrent_bwd, {name}: rel-L2 {rel:.2e}, max/RMS {mx:.2e}")
        assert rel <= TOL_REL and mx <= TOL_MAX, (name, rel, mx)
    cu = p.cu_seqlens_host
    for n, h in [(0, 0), (3, 11)]:
        a, b = cu[n], cu[n + 1]
        sl = lambda x: x[a:b, h:h + 1].cpu()
        ref = oracle.backward(sl(p.q), sl(p.k), sl(p.v), sl(p.z), sl(p.beta), [0, b - a], None,
                              sl(d_out), d_fin[n:n + 1, h:h + 1].cpu())
        mine = [g[a:b, h:h + 1] for g in got[:5]] + [got[5][n:n + 1, h:h + 1]]
        _compare(mine, ref, f"prefill workload ({n}, {h})")


def test_chunk_backward_matches_recurrent_on_varlen_workload():
    """The bench's varlen workload (64 sequences of 256..8192 tokens, 32 heads,
    initial state) in one launch: every gradient tensor against the per-token
    fp32 reverse mode on the GPU (itself held to the oracle at 1e-4), with the
    cotangents the bench draws."""
    p = workloads.prefill_workload("varlen", device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(99)
    H = p.meta["num_heads"]
    d_out = torch.randn(p.v.shape, device=DEV, generator=g).to(p.q.dtype)
    d_fin = torch.randn((p.num_seqs, H, 128, 128), device=DEV, generator=g)
    got = _run(p, d_out, d_fin)
    ref = kda.recurrent_bwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state, d_out,
                            d_fin, cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    for name, x, r in zip(NAMES, got, ref):
        diff = (x - r).double()
        rel = float(torch.linalg.vector_norm(diff) / torch.linalg.vector_norm(r.double()))
        rms = float(torch.sqrt(torch.mean(r.double() ** 2)))
        mx = float(diff.abs().max()) / rms
        print(f"varlen workload vs recurrent_bwd, {name}: rel-L2 {rel:.2e}, max/RMS {mx:.2e}")
        assert rel <= TOL_REL and mx <= TOL_MAX, (name, rel, mx)
        del diff
    del got, ref
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fn", ["recurrent_bwd", "chunk_bwd"])
def test_backward_device_lengths_beyond_the_host_plan(fn):
    """The workspace is planned from the host copy of cu_seqlens; a device copy
    with a longer sequence than planned makes the kernel skip that sequence
    (no workspace access past the plan), record KDA_ERR_DEVICE_CHECK, and leave
    the context usable: the next call with matching offsets is correct."""
    p = workloads.random_problem([20, 20], 1, 128, 128, torch.bfloat16, init_std=0.1, seed=31,
                                 device=DEV)
    d_out, d_fin = _cotangents(p, 12)
    f = getattr(kda, fn)
    bad = torch.tensor([0, 5, 40], dtype=torch.int32, device=DEV)  # sequence 1: 35 > 20 tokens
    assert kda.get_device_error() == 0
    f(p.q, p.k, p.v, p.z, p.beta, bad, p.initial_state, d_out, d_fin,
      cu_seqlens_host=p.cu_seqlens_host)
    assert kda.get_device_error() == 5
    assert kda.get_device_error() == 0  # cleared by the read
    got = f(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state, d_out, d_fin,
            cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    ref = oracle.backward(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                          d_out, d_fin)
    _compare(got, ref, f"{fn} after a device check")
