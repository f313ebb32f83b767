"""Context parallelism on the GPU kernels, the ranks emulated in one process
on one GPU (stacking the summaries stands in for the all-gather; no kernel
waits on another): kda_chunk_fwd_summary against the oracle's affine
summary, kda_state_scan against the oracle's scan, and the whole scheme --
summaries of every rank's pieces, scan, prefill of each piece from its
entering state -- against one pass over the whole sequences."""
import numpy as np
import pytest
import torch

import linear_attention_layer_gb300 as kda
import oracle
import workloads
from linear_attention_layer_gb300 import context_parallel as cp
from tests.parity import assert_close, device_compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("per_head_gate", [False, True])
def test_summary_matches_oracle(split, per_head_gate):
    """Slow decay (z ~ N(-4, 0.5): about e^-0.09 per token), so that M stays
    well inside the fp32 range over 700 tokens and can be compared element by
    element."""
    p = workloads.random_problem([700, 0, 130, 1], 2, 128, 128, torch.bfloat16, z_mean=-4.0,
                                 z_std=0.5, seed=51, device=DEV)
    z = p.z[:, :, 0].contiguous() if per_head_gate else p.z
    A = torch.tensor([0.3, -0.6], device=DEV)
    ws = "auto" if split else None
    if split:
        assert kda.chunk_fwd_summary_workspace_size(4, p.total_tokens, 2, 128, 128,
                                                    torch.bfloat16, p.cu_seqlens_host) > 0
    m, s = kda.chunk_fwd_summary(p.q, p.k, p.v, z, p.beta, p.cu_seqlens, p.cu_seqlens_host,
                                 workspace=ws, a_log=A)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    zo = z.cpu()[:, :, None].expand(-1, -1, 128).contiguous() if per_head_gate else p.z
    rm, rs = oracle.affine_summary(p.q, p.k, p.v, zo, p.beta, p.cu_seqlens_host, a_log=A.cpu())
    assert_close(s, rs, torch.bfloat16, "offset state S~")
    assert_close(m, rm, torch.bfloat16, "transition M")
    # the empty sequence: identity and zero
    assert torch.equal(m[1], torch.eye(128, device=DEV).expand(2, 128, 128))
    assert torch.equal(s[1], torch.zeros_like(s[1]))


@pytest.mark.parametrize("split", [False, True])
def test_summary_action_on_a_state(split):
    """Ordinary gates (z ~ N(0, 1.5)): M S_in + S~ equals the recurrence run
    from S_in (M's entries may underflow fp32 here -- the true values are
    below e^-300 -- which changes nothing the summary is used for)."""
    p = workloads.random_problem([700, 0, 130, 1], 2, 128, 128, torch.bfloat16, z_std=1.5,
                                 init_std=0.3, seed=53, device=DEV)
    m, s = kda.chunk_fwd_summary(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.cu_seqlens_host,
                                 workspace="auto" if split else None)
    got = torch.matmul(m.double(), p.initial_state.double()) + s.double()
    torch.cuda.synchronize()
    _, rf, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state)
    assert_close(got.cpu(), rf, torch.bfloat16, "M S_in + S~")


@pytest.mark.parametrize("dk,dv", [(32, 64), (64, 32), (128, 128)])
def test_state_scan_matches_oracle(dk, dv):
    g = torch.Generator(device=DEV).manual_seed(5)
    R, N, H = 3, 5, 2
    m = torch.randn((R, N, H, dk, dk), device=DEV, generator=g) / dk ** 0.5
    s = torch.randn((R, N, H, dk, dv), device=DEV, generator=g)
    s0 = torch.randn((N, H, dk, dv), device=DEV, generator=g)
    for count in range(R + 1):
        for init in (s0, None):
            got = kda.state_scan(m, s, init, count=count)
            ref = oracle.state_scan(m.cpu(), s.cpu(), None if init is None else init.cpu(),
                                    count=count)
            assert_close(got, ref, torch.float32, f"scan count={count}")
    x = s0.clone()
    kda.state_scan(m, s, x, out=x)  # in place
    torch.cuda.synchronize()
    assert_close(x, oracle.state_scan(m.cpu(), s.cpu(), s0.cpu()), torch.float32, "in place")


def _emulate(p, world, a_log=None):
    """Every rank's summary, scan and prefill, run one after the other."""
    bounds = cp.shard_bounds(p.cu_seqlens_host, world)
    pieces = []
    for r in range(world):
        idx, cu = [], [0]
        for n, b in enumerate(bounds):
            st = p.cu_seqlens_host[n]
            idx += list(range(st + b[r], st + b[r + 1]))
            cu.append(cu[-1] + b[r + 1] - b[r])
        it = torch.tensor(idx, dtype=torch.long, device=DEV)
        sel = lambda x: x.index_select(0, it).contiguous()
        pieces.append((it, cu, [sel(x) for x in (p.q, p.k, p.v, p.z, p.beta)]))
    ops = cp.LibraryOps()
    ms, ss = [], []
    for it, cu, xs in pieces:
        m, s = ops.summary(*xs, torch.tensor(cu, dtype=torch.int32, device=DEV), cu, a_log)
        ms.append(m)
        ss.append(s)
    ms, ss = torch.stack(ms), torch.stack(ss)
    out = torch.empty_like(p.v)
    fin = None
    for r, (it, cu, xs) in enumerate(pieces):
        entry = ops.scan(ms, ss, p.initial_state, r)
        o, fin = ops.prefill(*xs, torch.tensor(cu, dtype=torch.int32, device=DEV), cu, entry,
                             a_log)
        out.index_copy_(0, it, o)
    torch.cuda.synchronize()
    return out, fin


@pytest.mark.parametrize("world", [2, 3])
def test_context_parallel_emulated_matches_one_pass(world):
    p = workloads.random_problem([3000, 1000, 40, 0], 2, 128, 128, torch.bfloat16,
                                 init_std=0.1, seed=52, device=DEV)
    A = torch.tensor([0.5, -0.2], device=DEV)
    out, fin = _emulate(p, world, A)
    assert kda.get_device_error() == 0
    ro, rf, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host,
                                 p.initial_state, a_log=A.cpu())
    assert_close(out, ro, torch.bfloat16, f"{world} ranks out")
    assert_close(fin, rf, torch.bfloat16, f"{world} ranks final state")


def test_context_parallel_long_workload_four_ranks():
    """The slow-decay long-context workload (1 x 65536 tokens, 32 heads, z ~
    N(-2, 1)) cut over four emulated ranks equals the single-GPU prefill of
    the whole sequence."""
    p = workloads.prefill_workload("long_slow", device=DEV)
    out, fin = _emulate(p, 4)
    ref_o, ref_f = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, None,
                                 cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    for x, r, what, both in ((out, ref_o, "out", True), (fin, ref_f, "final", False)):
        rel, mx = device_compare(x, r, both_stored=both)
        print(f"4 emulated ranks vs one pass, {what}: rel-L2 {rel:.3e}, max/RMS {mx:.3e}")
        assert rel <= 1e-2 and mx <= 2e-2, (what, rel, mx)
