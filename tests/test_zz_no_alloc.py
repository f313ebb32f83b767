"""kda_chunk_fwd_noalloc: the chunked prefill for callers that cannot
allocate device memory (their HBM is owned by a host framework that reserved
it up front, or they run where cudaMalloc is not allowed or its implicit
synchronisation is too costly).  Its scratch for splitting long sequences is
an array inside the library, shared by every call.

These GPU tests call it through the C ABI and compare it with kda_chunk_fwd
given an explicitly allocated workspace, on two calls in a row with different
inputs (the second call starts from the first call's leftover scratch), and
on the long-context workload (the call takes the best split whose summaries
fit in the array, or none).  This file
is collected after the other test files on purpose."""
import os
import re

import pytest
import torch

import linear_attention_layer_gb300 as kda
import workloads
from tests.parity import assert_close, device_compare

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEV = "cuda:0"


def _ws_bytes(p):
    return kda.chunk_fwd_workspace_size(p.num_seqs, p.total_tokens, p.meta["num_heads"],
                                        p.meta["dk"], p.meta["dv"], p.q.dtype, p.cu_seqlens_host)


def test_binding_constant_matches_header():
    text = open(os.path.join(ROOT, "include", "kda.h"), encoding="utf-8").read()
    m = re.search(r"#define KDA_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == kda.NOALLOC_SCRATCH_BYTES


@pytest.mark.gpu
def test_noalloc_matches_chunk_fwd_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    for seed in (41, 42):
        p = workloads.random_problem([3000, 700, 64], 3, 128, 128, torch.bfloat16, init_std=0.1,
                                     seed=seed, device=DEV)
        need = _ws_bytes(p)
        assert 0 < need <= kda.NOALLOC_SCRATCH_BYTES  # the split runs and fits
        ref_out, ref_fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens,
                                         p.initial_state, cu_seqlens_host=p.cu_seqlens_host,
                                         workspace=torch.empty(need, dtype=torch.uint8,
                                                               device=DEV))
        out = torch.empty_like(ref_out)
        fin = torch.empty_like(ref_fin)
        kda.chunk_fwd_noalloc(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                              out=out, final_state=fin, cu_seqlens_host=p.cu_seqlens_host)
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        assert_close(out, ref_out, torch.bfloat16, f"noalloc out (seed {seed})", both_stored=True)
        assert_close(fin, ref_fin, torch.bfloat16, f"noalloc final state (seed {seed})")


@pytest.mark.gpu
def test_noalloc_long_sequence():
    """The long-context workload (1 x 65536 tokens, 32 heads) on two calls in
    a row: the call takes the best split whose summaries fit in the array
    (or none) -- nothing allocated -- and its results equal kda_chunk_fwd's
    with a full workspace."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    p = workloads.prefill_workload("long", device=DEV)
    need = _ws_bytes(p)
    assert need > 0
    ref_out, ref_fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, None,
                                     cu_seqlens_host=p.cu_seqlens_host,
                                     workspace=torch.empty(need, dtype=torch.uint8, device=DEV))
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        kda.chunk_fwd_noalloc(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, None, out=out,
                              final_state=fin, cu_seqlens_host=p.cu_seqlens_host)
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        for x, r, what, both in ((out, ref_out, "out", True), (fin, ref_fin, "final", False)):
            rel, mx = device_compare(x, r, both_stored=both)
            assert rel <= 1e-2 and mx <= 2e-2, f"noalloc long {what}: rel-L2 {rel:.3e}, max {mx:.3e}"
