"""kda_chunk_fwd_fused: the chunked prefill over raw q, k with the short
convolution + Swish fused into the tensor-core kernel, against the oracle
composition (oracle.short_conv of q and k from each sequence's convolution
state, then the fp64 recurrence on its unrounded results), and against the
two separate calls (kda_short_conv, then kda_chunk_fwd).  The convolution states
left behind are each sequence's last raw inputs, compared bit for bit."""
import numpy as np
import pytest
import torch

import linear_attention_layer_gb300 as kda
import oracle
import workloads
from tests.parity import WholeTensorError, assert_close, problem_pieces, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.load()
    torch.cuda.set_device(0)


def _conv_inputs(N, H, W, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    f32 = dict(dtype=torch.float32, device=DEV, generator=g)
    wq = torch.randn((H, 128, W), **f32) * 0.6
    wk = torch.randn((H, 128, W), **f32) * 0.6
    sq = torch.randn((N, H, 128, max(W - 1, 0)), **f32)
    sk = torch.randn((N, H, 128, max(W - 1, 0)), **f32)
    return wq, wk, sq, sk


def _oracle(p, wq, wk, sq, sk, z=None, a_log=None):
    """The composition the fused call computes: the convolution + Swish
    (fp64), then the fp64 recurrence on its unrounded results."""
    cu = p.cu_seqlens_host
    W = wq.shape[-1]
    qy, fq = oracle.short_conv(p.q, wq, cu, sq.cpu() if W > 1 else None)
    ky, fk = oracle.short_conv(p.k, wk, cu, sk.cpu() if W > 1 else None)
    o, f, _ = oracle.recurrent(qy, ky, p.v, p.z if z is None else z, p.beta, cu,
                               p.initial_state, a_log=a_log)
    return o, f, fq, fk


LENS = [1, 2, 3, 15, 64, 65, 0, 130, 200]


@pytest.mark.parametrize("W", [4, 3, 2, 1])
def test_fused_prefill_matches_oracle(W):
    p = workloads.random_problem(LENS, 2, 128, 128, torch.bfloat16, init_std=0.1, seed=80 + W,
                                 device=DEV, normalize_qk=False)
    wq, wk, sq, sk = _conv_inputs(len(LENS), 2, W, 90 + W)
    sq0, sk0 = sq.clone(), sk.clone()
    out, fin = kda.chunk_fwd_fused(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                   conv_weight_q=wq, conv_weight_k=wk,
                                   conv_state_q=sq if W > 1 else None,
                                   conv_state_k=sk if W > 1 else None,
                                   cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    ro, rf, fq, fk = _oracle(p, wq, wk, sq0, sk0)
    assert_close(out, ro, torch.bfloat16, f"W={W} out")
    assert_close(fin, rf, torch.bfloat16, f"W={W} final state")
    if W > 1:
        assert torch.equal(sq.cpu(), torch.from_numpy(fq).float())
        assert torch.equal(sk.cpu(), torch.from_numpy(fk).float())


def test_fused_prefill_split_per_head_gate_and_log_scale():
    """Long sequences split across SMs (a segment's first halo comes from the
    raw inputs before it), one gate per head and the gate log-scale."""
    lens = [3000, 700, 2]
    p = workloads.random_problem(lens, 2, 128, 128, torch.bfloat16, init_std=0.1, seed=85,
                                 device=DEV, normalize_qk=False)
    assert kda.chunk_fwd_workspace_size(3, p.total_tokens, 2, 128, 128, torch.bfloat16,
                                        p.cu_seqlens_host) > 0
    wq, wk, sq, sk = _conv_inputs(3, 2, 4, 86)
    sq0, sk0 = sq.clone(), sk.clone()
    zh = p.z[:, :, 0].contiguous()
    A = torch.tensor([0.4, -0.3], device=DEV)
    out, fin = kda.chunk_fwd_fused(p.q, p.k, p.v, zh, p.beta, p.cu_seqlens, p.initial_state,
                                   conv_weight_q=wq, conv_weight_k=wk, conv_state_q=sq,
                                   conv_state_k=sk, cu_seqlens_host=p.cu_seqlens_host,
                                   workspace="auto", a_log=A)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    zo = zh.cpu()[:, :, None].expand(-1, -1, 128).contiguous()
    ro, rf, fq, fk = _oracle(p, wq, wk, sq0, sk0, z=zo, a_log=A.cpu())
    assert_close(out, ro, torch.bfloat16, "split out")
    assert_close(fin, rf, torch.bfloat16, "split final state")
    assert torch.equal(sq.cpu(), torch.from_numpy(fq).float())


def test_fused_prefill_continues_a_split_sequence():
    """A sequence cut in two calls, the convolution and KDA states carried
    from the first to the second, equals one call over the whole sequence."""
    p = workloads.random_problem([500], 2, 128, 128, torch.bfloat16, init_std=0.1, seed=87,
                                 device=DEV, normalize_qk=False)
    wq, wk, sq, sk = _conv_inputs(1, 2, 4, 88)
    sq2, sk2 = sq.clone(), sk.clone()
    out, fin = kda.chunk_fwd_fused(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                   conv_weight_q=wq, conv_weight_k=wk, conv_state_q=sq,
                                   conv_state_k=sk)
    t = 203
    sl = lambda x, a, b: x[a:b].contiguous()
    cu = lambda n: torch.tensor([0, n], dtype=torch.int32, device=DEV)
    oa, fa = kda.chunk_fwd_fused(*(sl(x, 0, t) for x in (p.q, p.k, p.v, p.z, p.beta)), cu(t),
                                 p.initial_state, conv_weight_q=wq, conv_weight_k=wk,
                                 conv_state_q=sq2, conv_state_k=sk2)
    ob, fb = kda.chunk_fwd_fused(*(sl(x, t, 500) for x in (p.q, p.k, p.v, p.z, p.beta)),
                                 cu(500 - t), fa, conv_weight_q=wq, conv_weight_k=wk,
                                 conv_state_q=sq2, conv_state_k=sk2)
    torch.cuda.synchronize()
    assert_close(torch.cat([oa, ob]), out, torch.bfloat16, "two calls vs one", both_stored=True)
    assert_close(fb, fin, torch.bfloat16, "final state")
    assert torch.equal(sq2, sq) and torch.equal(sk2, sk)


def test_fused_prefill_full_prefill_workload():
    """The 4 x 4096-token, 16-head workload through the fused call, every
    output and final state against the oracle composition."""
    p = workloads.prefill_workload("prefill", device=DEV)
    wq, wk, sq, sk = _conv_inputs(p.num_seqs, 16, 4, 84)
    sq0, sk0 = sq.clone(), sk.clone()
    out, fin = kda.chunk_fwd_fused(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, None,
                                   conv_weight_q=wq, conv_weight_k=wk, conv_state_q=sq,
                                   conv_state_k=sk, cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    ro, rf, fq, fk = _oracle(p, wq, wk, sq0, sk0)
    print("fused prefill 4x4096x16 out rel-L2", assert_close(out, ro, torch.bfloat16, "out"))
    assert_close(fin, rf, torch.bfloat16, "final state")
    assert torch.equal(sq.cpu(), torch.from_numpy(fq).float())


def test_fused_prefill_full_varlen_workload():
    """The bench workload (64 sequences of 256..8192 tokens, 32 heads, initial
    states) through the fused call, every output and final state against the
    oracle composition (run piece by piece), and against the separate calls:
    kda_short_conv hands the convolved q, k over in bf16 where the fused call
    keeps fp16, so the two are compared by relative L2 error only (the max
    error of that comparison measures the bf16 rounding of q and k)."""
    p = workloads.prefill_workload("varlen", device=DEV)
    H = p.meta["num_heads"]
    wq, wk, sq, sk = _conv_inputs(p.num_seqs, H, 4, 89)
    sq0, sk0 = sq.clone(), sk.clone()
    o_f, f_f = kda.chunk_fwd_fused(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                   conv_weight_q=wq, conv_weight_k=wk, conv_state_q=sq,
                                   conv_state_k=sk, cu_seqlens_host=p.cu_seqlens_host)
    yq, fq = kda.short_conv(p.q, wq, p.cu_seqlens, sq0)
    yk, fk = kda.short_conv(p.k, wk, p.cu_seqlens, sk0)
    o_s, f_s = kda.chunk_fwd(yq, yk, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert torch.equal(sq, fq) and torch.equal(sk, fk)
    assert rel_l2(o_f, o_s) <= 1e-2 and rel_l2(f_f, f_s) <= 1e-2
    cu = p.cu_seqlens_host
    acc_o, acc_f = WholeTensorError(H, torch.bfloat16), WholeTensorError(H)
    wqc, wkc = wq.cpu(), wk.cpu()
    for (n0, n1), _ in problem_pieces(p):
        a, b = cu[n0], cu[n1]
        lcu = [x - a for x in cu[n0:n1 + 1]]
        qy, _ = oracle.short_conv(p.q[a:b].cpu(), wqc, lcu, sq0[n0:n1].cpu())
        ky, _ = oracle.short_conv(p.k[a:b].cpu(), wkc, lcu, sk0[n0:n1].cpu())
        ro, rf, _ = oracle.recurrent(qy, ky, p.v[a:b].cpu(), p.z[a:b].cpu(), p.beta[a:b].cpu(),
                                     lcu, p.initial_state[n0:n1].cpu())
        acc_o.add(o_f[a:b].cpu(), ro, head_axis=1)
        acc_f.add(f_f[n0:n1].cpu(), rf, head_axis=1)
    print(acc_o.check(torch.bfloat16, "fused varlen out"))
    print(acc_f.check(torch.bfloat16, "fused varlen final state"))


def test_fused_prefill_checkpoints():
    """State checkpoints every 64 tokens through the fused call: each equals
    the oracle composition's final state of that prefix."""
    lens = [64, 200, 0, 130]
    p = workloads.random_problem(lens, 2, 128, 128, torch.bfloat16, init_std=0.1, seed=91,
                                 device=DEV, normalize_qk=False)
    wq, wk, sq, sk = _conv_inputs(len(lens), 2, 4, 92)
    sq0, sk0 = sq.clone(), sk.clone()
    out, fin, ck = kda.chunk_fwd_fused(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                       conv_weight_q=wq, conv_weight_k=wk, conv_state_q=sq,
                                       conv_state_k=sk, cu_seqlens_host=p.cu_seqlens_host,
                                       checkpoint_every=64)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert ck.shape[0] == 1 + 3 + 0 + 2
    cu = p.cu_seqlens_host
    i = 0
    for n in range(len(lens)):
        for j in range(1, lens[n] // 64 + 1):
            a, b = cu[n], cu[n] + 64 * j
            qy, _ = oracle.short_conv(p.q[a:b].cpu(), wq.cpu(), [0, b - a], sq0[n:n + 1].cpu())
            ky, _ = oracle.short_conv(p.k[a:b].cpu(), wk.cpu(), [0, b - a], sk0[n:n + 1].cpu())
            _, rf, _ = oracle.recurrent(qy, ky, p.v[a:b].cpu(), p.z[a:b].cpu(), p.beta[a:b].cpu(),
                                        [0, b - a], p.initial_state[n:n + 1].cpu())
            assert_close(ck[i], rf[0], torch.bfloat16, f"checkpoint {i}")
            i += 1
