"""``kda_chunk_fwd_host``: the prefill over host buffers, with the batch cut
into groups whose copies overlap the kernels.  Each group is one launch of the
same kernel over the same sequences, so the results must equal
``kda_chunk_fwd`` on device copies of the data bit for bit (no sequence is
long enough here for the device path to split it); one case is also checked
against the fp64 oracle."""
import pytest
import torch

import linear_attention_layer_gb300 as kda
import oracle
import workloads
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.load()
    torch.cuda.set_device(0)


def _host(t):
    return None if t is None else t.cpu().pin_memory()


@pytest.mark.parametrize("groups", [1, 3, 8, 100])
@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_host_prefill_equals_device_prefill(groups, dtype, d):
    lens = [300, 1, 0, 64, 65, 129, 17, 500, 2, 63]
    p = workloads.random_problem(lens, 3, d, d, dtype, z_std=1.5, init_std=0.2, seed=31,
                                 device=DEV)
    ref_out, ref_fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                     cu_seqlens_host=p.cu_seqlens_host)
    out, fin = kda.chunk_fwd_host(_host(p.q), _host(p.k), _host(p.v), _host(p.z), _host(p.beta),
                                  p.cu_seqlens_host, _host(p.initial_state), groups=groups)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out.cpu())
    assert torch.equal(fin, ref_fin.cpu())
    assert kda.get_device_error() == 0


def test_host_prefill_no_state_gate_scale_per_head_gate_and_oracle():
    p = workloads.random_problem([200, 70, 9], 2, 128, 128, torch.bfloat16, seed=32, device=DEV)
    a_log = torch.tensor([0.4, -0.8], dtype=torch.float32, device=DEV)
    zh = p.z[..., 0].contiguous()  # one gate per head
    for z in (p.z, zh):
        ref_out, _ = kda.chunk_fwd(p.q, p.k, p.v, z, p.beta, p.cu_seqlens, None,
                                   cu_seqlens_host=p.cu_seqlens_host, a_log=a_log,
                                   output_final_state=False)
        out, fin = kda.chunk_fwd_host(_host(p.q), _host(p.k), _host(p.v), _host(z),
                                      _host(p.beta), p.cu_seqlens_host, None, groups=2,
                                      a_log=a_log, output_final_state=False)
        assert fin is None
        assert torch.equal(out, ref_out.cpu())
    ro, _, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, None,
                                a_log=a_log.cpu().numpy())
    out, _ = kda.chunk_fwd_host(_host(p.q), _host(p.k), _host(p.v), _host(p.z), _host(p.beta),
                                p.cu_seqlens_host, None, groups=3, a_log=a_log)
    assert_close(out, ro, torch.bfloat16, "out")


def test_host_prefill_empty_sequences_keep_their_state():
    p = workloads.random_problem([0, 5, 0], 2, 128, 128, torch.bfloat16, init_std=0.2, seed=33,
                                 device=DEV)
    out, fin = kda.chunk_fwd_host(_host(p.q), _host(p.k), _host(p.v), _host(p.z), _host(p.beta),
                                  p.cu_seqlens_host, _host(p.initial_state), groups=3)
    ref_out, ref_fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                     cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out.cpu()) and torch.equal(fin, ref_fin.cpu())
    assert torch.equal(fin[0], p.initial_state[0].cpu()) and torch.equal(fin[2], p.initial_state[2].cpu())
