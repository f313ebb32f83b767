"""GPU parity: the libkda kernels (through the C ABI) against the fp64 oracle
on the same seeded inputs, element by element, with the tolerances of
tests/parity.py.  Small cases and the full-size workloads alike compare every output and every
final state."""
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


def _check_all(p, out, fin, io_dtype):
    ro, rf, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state)
    assert_close(out, ro, io_dtype, "out")
    assert_close(fin, rf, io_dtype, "final_state")


# ----------------------------------------------------------- small cases --

RAGGED = [1, 15, 16, 17, 0, 63, 65, 130]


@pytest.mark.parametrize("entry", ["chunk_fwd", "recurrent_fwd"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
def test_prefill_small_ragged(entry, dtype, dk, dv):
    p = workloads.random_problem(RAGGED, 3, dk, dv, dtype, z_std=1.5, init_std=0.1, seed=5,
                                 device=DEV)
    fn = getattr(kda, entry)
    out, fin = fn(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                  cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    _check_all(p, out, fin, dtype)
    assert kda.get_device_error() == 0


def test_tiny_workload_fp32():
    """B=1, H=1, T=64, dk=dv=32 in fp32: relative L2 <= 1e-4."""
    p = workloads.prefill_workload("tiny", device=DEV)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, None,
                             cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    _check_all(p, out, fin, torch.float32)


@pytest.mark.parametrize("z_mean", [-2.0, 2.0, 6.0])
def test_prefill_decay_extremes(z_mean):
    """Gate logits near saturation (16-token sums close to -80) and slow decay."""
    p = workloads.random_problem([300, 77], 2, 128, 128, torch.bfloat16, z_mean=z_mean,
                                 init_std=0.5, seed=7, device=DEV)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    _check_all(p, out, fin, torch.bfloat16)


def test_no_initial_state_no_final_state():
    p = workloads.random_problem([40, 9], 2, 64, 64, torch.float32, seed=8, device=DEV)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, None,
                             output_final_state=False)
    torch.cuda.synchronize()
    assert fin is None
    ro, _, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, None)
    assert_close(out, ro, torch.float32, "out")


def test_final_state_may_alias_initial_state():
    p = workloads.random_problem([50, 33, 0], 2, 128, 128, torch.bfloat16, init_std=0.1, seed=9,
                                 device=DEV)
    s0 = p.initial_state.clone()
    ro, rf, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, s0)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             final_state=p.initial_state)
    torch.cuda.synchronize()
    assert fin.data_ptr() == p.initial_state.data_ptr()
    assert_close(out, ro, torch.bfloat16, "out")
    assert_close(fin, rf, torch.bfloat16, "final_state")


def test_prefix_split_matches_whole_run():
    """final_state of tokens [0, t) fed back as initial_state of [t, T) equals
    one pass over [0, T) (prefix reuse)."""
    p = workloads.random_problem([500], 4, 128, 128, torch.bfloat16, init_std=0.1, seed=10,
                                 device=DEV)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state)
    t = 203
    cu_a = torch.tensor([0, t], dtype=torch.int32, device=DEV)
    cu_b = torch.tensor([0, 500 - t], dtype=torch.int32, device=DEV)
    sl = lambda x, a, b: x[a:b].contiguous()
    oa, fa = kda.chunk_fwd(sl(p.q, 0, t), sl(p.k, 0, t), sl(p.v, 0, t), sl(p.z, 0, t),
                           sl(p.beta, 0, t), cu_a, p.initial_state)
    ob, fb = kda.chunk_fwd(sl(p.q, t, 500), sl(p.k, t, 500), sl(p.v, t, 500), sl(p.z, t, 500),
                           sl(p.beta, t, 500), cu_b, fa)
    torch.cuda.synchronize()
    assert rel_l2(torch.cat([oa, ob]), out) <= 1e-2
    assert rel_l2(fb, fin) <= 1e-2


def test_chunked_and_recurrent_gpu_paths_agree():
    p = workloads.random_problem([1000, 257, 3], 4, 128, 128, torch.bfloat16, init_std=0.1,
                                 seed=11, device=DEV)
    oc, fc = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                           cu_seqlens_host=p.cu_seqlens_host)
    orr, fr = kda.recurrent_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state)
    torch.cuda.synchronize()
    assert_close(oc, orr, torch.bfloat16, "out chunk vs recurrent", both_stored=True)
    assert_close(fc, fr, torch.bfloat16, "final chunk vs recurrent")


def test_zero_tokens_and_zero_length_sequences():
    p = workloads.random_problem([0, 0], 2, 64, 64, torch.bfloat16, init_std=0.1, seed=12,
                                 device=DEV)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state)
    torch.cuda.synchronize()
    assert out.shape == (0, 2, 64)
    assert torch.equal(fin, p.initial_state)


def test_bad_device_cu_seqlens_sets_error_word():
    """The host copy is absent, so only the kernel can see the out-of-range
    offset: it skips that sequence, records KDA_ERR_DEVICE_CHECK, and the
    context stays usable."""
    p = workloads.random_problem([20, 20], 1, 64, 64, torch.bfloat16, seed=13, device=DEV)
    bad = torch.tensor([0, 20, 999], dtype=torch.int32, device=DEV)
    assert kda.get_device_error() == 0
    kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, bad, None)
    assert kda.get_device_error() == 5
    assert kda.get_device_error() == 0  # cleared by the read
    out, _ = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, None)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


# ---------------------------------------------------------------- decode --

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 128)])
def test_decode_steps_small(dtype, dk, dv):
    d = workloads.decode_workload(5, 3, dk, dv, steps=6, io_dtype=dtype, device=DEV, seed=3)
    S = d.state.clone()
    s_ref = d.state.cpu()
    for t in range(6):
        o = kda.decode_step(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], S)
        torch.cuda.synchronize()
        ro, s_ref = oracle.decode_step(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], s_ref)
        assert_close(o, ro, dtype, f"decode out step {t}")
    assert_close(S, s_ref, dtype, "decode state")


def test_decode_chain_equals_prefill():
    """T decode steps on one request equal a T-token prefill (GPU paths)."""
    T = 48
    p = workloads.random_problem([T], 2, 128, 128, torch.bfloat16, init_std=0.1, seed=14,
                                 device=DEV)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state)
    S = p.initial_state.clone()
    outs = []
    for t in range(T):
        sl = lambda x: x[t:t + 1].contiguous()
        outs.append(kda.decode_step(sl(p.q), sl(p.k), sl(p.v), sl(p.z), sl(p.beta), S))
    torch.cuda.synchronize()
    assert_close(torch.cat(outs), out, torch.bfloat16, "decode chain vs chunk out",
                 both_stored=True)
    assert_close(S, fin, torch.bfloat16, "decode chain vs chunk state")


# ------------------------------------------------- gate log-scale A -------

@pytest.mark.parametrize("entry,dtype,dk,dv", [
    ("chunk_fwd", torch.bfloat16, 128, 128),   # tensor-core kernel
    ("chunk_fwd", torch.float32, 64, 32),      # CUDA-core chunked kernel
    ("recurrent_fwd", torch.bfloat16, 128, 64),
    ("chunk_fwd_noalloc", torch.bfloat16, 128, 128),
])
def test_gate_log_scale(entry, dtype, dk, dv):
    """g = -5 sigmoid(e^{A_h} z) with a different A per head, against the oracle
    given the same A."""
    p = workloads.random_problem(RAGGED, 3, dk, dv, dtype, z_std=1.5, init_std=0.1, seed=11,
                                 device=DEV)
    A = torch.tensor([0.6, -1.2, 1.7], dtype=torch.float32)
    out, fin = getattr(kda, entry)(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                   cu_seqlens_host=p.cu_seqlens_host, a_log=A.to(DEV))
    torch.cuda.synchronize()
    ro, rf, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state,
                                 a_log=A)
    assert_close(out, ro, dtype, "out")
    assert_close(fin, rf, dtype, "final_state")
    # and A really acts: without it the result moves well outside the tolerance
    ro0, _, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state)
    assert rel_l2(out, ro0) > 10 * rel_l2(out, ro)
    assert kda.get_device_error() == 0


def test_decode_gate_log_scale():
    d = workloads.decode_workload(4, 3, 128, 128, steps=3, io_dtype=torch.bfloat16, device=DEV,
                                  seed=4)
    A = torch.tensor([-0.8, 0.3, 2.0], dtype=torch.float32)
    S = d.state.clone()
    s_ref = d.state.cpu()
    for t in range(3):
        o = kda.decode_step(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], S, a_log=A.to(DEV))
        torch.cuda.synchronize()
        ro, s_ref = oracle.decode_step(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], s_ref, a_log=A)
        assert_close(o, ro, torch.bfloat16, f"decode out step {t}")
    assert_close(S, s_ref, torch.bfloat16, "decode state")


# ------------------------------------------- one gate per head (scalar alpha) --

@pytest.mark.parametrize("entry,dtype,dk,dv", [
    ("chunk_fwd", torch.bfloat16, 128, 128),   # tensor-core kernel
    ("chunk_fwd", torch.float32, 32, 64),      # CUDA-core chunked kernel
    ("recurrent_fwd", torch.bfloat16, 64, 128),
])
def test_gate_per_head(entry, dtype, dk, dv):
    """z [T, H]: every key channel of a head gets the same retention.  The
    oracle runs the per-channel gate with that logit broadcast over dk."""
    p = workloads.random_problem(RAGGED, 3, dk, dv, dtype, z_std=1.5, init_std=0.1, seed=17,
                                 device=DEV)
    zh = p.z[:, :, 0].contiguous()  # [T, H]
    A = torch.tensor([0.2, -0.9, 1.1])
    out, fin = getattr(kda, entry)(p.q, p.k, p.v, zh, p.beta, p.cu_seqlens, p.initial_state,
                                   cu_seqlens_host=p.cu_seqlens_host, a_log=A.to(DEV))
    torch.cuda.synchronize()
    zb = zh.cpu()[:, :, None].expand(-1, -1, dk).contiguous()
    ro, rf, _ = oracle.recurrent(p.q, p.k, p.v, zb, p.beta, p.cu_seqlens_host, p.initial_state,
                                 a_log=A)
    assert_close(out, ro, dtype, "out")
    assert_close(fin, rf, dtype, "final_state")
    assert kda.get_device_error() == 0


def test_gate_per_head_decode_and_window():
    d = workloads.decode_workload(4, 2, 128, 128, steps=2, io_dtype=torch.bfloat16, device=DEV,
                                  seed=8)
    S = d.state.clone()
    s_ref = d.state.cpu()
    for t in range(2):
        zh = d.z[t][:, :, 0].contiguous()
        o = kda.decode_step(d.q[t], d.k[t], d.v[t], zh, d.beta[t], S)
        torch.cuda.synchronize()
        ro, s_ref = oracle.decode_step(d.q[t], d.k[t], d.v[t],
                                       zh.cpu()[:, :, None].expand(-1, -1, 128), d.beta[t],
                                       s_ref)
        assert_close(o, ro, torch.bfloat16, f"decode out step {t}")
    assert_close(S, s_ref, torch.bfloat16, "decode state")
    q, k, v, z, beta, state = _window_inputs(3, 4, 2, 128, 128, torch.bfloat16, 24)
    zh = z[..., 0].contiguous()  # [B, W, H]
    out = kda.decode_window(q, k, v, zh, beta, state)
    ref, _ = _oracle_window(q, k, v, zh[..., None].expand(-1, -1, -1, 128).contiguous(), beta,
                            state, [4] * 3)
    assert_close(out, np.stack(ref), torch.bfloat16, "window outputs")


# ------------------------------------------------ speculative decoding -----

def _window_inputs(B, W, H, dk, dv, dtype, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    f32 = dict(dtype=torch.float32, device=DEV, generator=g)
    unit = lambda x: x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)
    q = unit(torch.randn((B, W, H, dk), **f32)).to(dtype)
    k = unit(torch.randn((B, W, H, dk), **f32)).to(dtype)
    v = torch.randn((B, W, H, dv), **f32).to(dtype)
    z = torch.randn((B, W, H, dk), **f32)
    beta = torch.sigmoid(torch.randn((B, W, H), **f32))
    state = torch.randn((B, H, dk, dv), **f32) * 0.1
    return q, k, v, z, beta, state


def _oracle_window(q, k, v, z, beta, state, ntok, a_log=None):
    """Per request b: its first ntok[b] drafts as a sequence from state[b]."""
    B, W = q.shape[:2]
    outs, fins = [], []
    for b in range(B):
        n = int(ntok[b])
        o, f, _ = oracle.recurrent(q[b, :n].cpu(), k[b, :n].cpu(), v[b, :n].cpu(),
                                   z[b, :n].cpu(), beta[b, :n].cpu(), [0, n],
                                   state[b:b + 1].cpu(), a_log=a_log)
        outs.append(o)
        fins.append(f[0])
    return outs, np.stack(fins)


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 32),
                                         (torch.float32, 32, 64), (torch.bfloat16, 128, 64),
                                         (torch.bfloat16, 32, 128), (torch.float32, 128, 32)])
def test_decode_window_outputs_and_state_untouched(dtype, dk, dv):
    B, W, H = 5, 4, 3
    q, k, v, z, beta, state = _window_inputs(B, W, H, dk, dv, dtype, 21)
    A = torch.tensor([0.3, -0.5, 1.0])
    before = state.clone()
    out = kda.decode_window(q, k, v, z, beta, state, a_log=A.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(state, before)
    ref, _ = _oracle_window(q, k, v, z, beta, before, [W] * B, a_log=A)
    assert_close(out, np.stack(ref), dtype, "window outputs")
    assert kda.get_device_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_replay_applies_accepted_prefix(dtype):
    B, W, H, dk, dv = 6, 5, 2, 128, 64
    q, k, v, z, beta, state = _window_inputs(B, W, H, dk, dv, dtype, 22)
    acc = [0, 5, 1, 3, 2, 4]
    before = state.clone()
    kda.decode_replay(q, k, v, z, beta, torch.tensor(acc, dtype=torch.int32, device=DEV), state)
    torch.cuda.synchronize()
    _, ref = _oracle_window(q, k, v, z, beta, before, acc)
    assert torch.equal(state[0], before[0])   # nothing accepted: state untouched
    assert_close(state, ref, dtype, "replayed states")
    assert kda.get_device_error() == 0


def _misaligned(x, elems=1):
    """x's values in a contiguous tensor whose data starts `elems` elements
    past an allocation's start (not 16-byte aligned)."""
    buf = torch.empty(x.numel() + elems, dtype=x.dtype, device=x.device)
    y = buf[elems:].view(x.shape)
    y.copy_(x)
    return y


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_window_inputs_not_16_byte_aligned(dtype):
    """q, k, v, z that start off a 16-byte boundary (element-wise input
    copies) give the results of the aligned call bit for bit."""
    B, W, H, dk, dv = 4, 3, 2, 128, 128
    q, k, v, z, beta, state = _window_inputs(B, W, H, dk, dv, dtype, 27)
    acc = torch.tensor([0, 3, 1, 2], dtype=torch.int32, device=DEV)
    s1, s2 = state.clone(), state.clone()
    o1 = kda.decode_replay_window((q, k, v, z, beta), acc, q, k, v, z, beta, s1)
    mq, mk, mv, mz = (_misaligned(x) for x in (q, k, v, z))
    assert all(x.data_ptr() % 16 for x in (mq, mk, mv, mz))
    o2 = kda.decode_replay_window((mq, mk, mv, mz, beta), acc, mq, mk, mv, mz, beta, s2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    ref, fins = _oracle_window(q, k, v, z, beta, state, acc.tolist())
    assert_close(s2, fins, dtype, "replayed states")
    assert kda.get_device_error() == 0


def test_draft_verify_replay_loop_equals_prefill_of_accepted_tokens():
    """Three rounds of window + replay; the final states equal a prefill over
    the accepted tokens only, and every window output the oracle's."""
    B, W, H, dk, dv = 4, 4, 2, 128, 128
    torch.manual_seed(0)
    state = torch.randn((B, H, dk, dv), device=DEV) * 0.1
    s0 = state.clone()
    accepted = [[] for _ in range(B)]
    rng = np.random.default_rng(5)
    for r in range(3):
        q, k, v, z, beta, _ = _window_inputs(B, W, H, dk, dv, torch.bfloat16, 30 + r)
        out = kda.decode_window(q, k, v, z, beta, state)
        ref, _ = _oracle_window(q, k, v, z, beta, state, [W] * B)
        assert_close(out, np.stack(ref), torch.bfloat16, f"round {r} outputs")
        acc = rng.integers(0, W + 1, size=B)
        kda.decode_replay(q, k, v, z, beta, torch.tensor(acc, dtype=torch.int32, device=DEV),
                          state)
        for b in range(B):
            accepted[b] += [(q[b, i], k[b, i], v[b, i], z[b, i], beta[b, i]) for i in range(acc[b])]
    torch.cuda.synchronize()
    for b in range(B):
        n = len(accepted[b])
        if n == 0:
            assert torch.equal(state[b], s0[b])
            continue
        cols = [torch.stack([t[j] for t in accepted[b]]).cpu() for j in range(5)]
        _, fin, _ = oracle.recurrent(*cols, [0, n], s0[b:b + 1].cpu())
        assert_close(state[b], fin[0], torch.bfloat16, f"request {b} after {n} accepted")


def test_fused_replay_window_equals_replay_then_window():
    """One launch per step (replay of the previous window's accepted prefix,
    then the new window's outputs) against the two separate calls."""
    B, W, H, dk, dv = 5, 3, 2, 128, 128
    torch.manual_seed(1)
    s_sep = torch.randn((B, H, dk, dv), device=DEV) * 0.1
    s_fused = s_sep.clone()
    prev = _window_inputs(B, W, H, dk, dv, torch.bfloat16, 40)[:5]
    kda.decode_window(*prev, s_sep)
    rng = np.random.default_rng(9)
    for r in range(3):
        nxt = _window_inputs(B, W + r, H, dk, dv, torch.bfloat16, 41 + r)[:5]
        acc = torch.tensor(rng.integers(0, W + 1, size=B), dtype=torch.int32, device=DEV)
        kda.decode_replay(*prev, acc, s_sep)
        o_sep = kda.decode_window(*nxt, s_sep)
        o_fused = kda.decode_replay_window(prev, acc, *nxt, s_fused)
        torch.cuda.synchronize()
        assert torch.equal(o_fused, o_sep)
        assert torch.equal(s_fused, s_sep)
        prev = nxt
        W = W + r
    assert kda.get_device_error() == 0


def test_speculative_decoding_many_units_streamed():
    """Enough (request, head) units (40 x 16 = 640) for the persistent kernel
    that streams the next unit's state in while applying the current one:
    the fused call equals the separate calls bit for bit, sampled requests
    equal the oracle, and a bad acceptance length leaves its request alone."""
    B, W, H, dk, dv = 40, 4, 16, 128, 128
    torch.manual_seed(2)
    s_sep = torch.randn((B, H, dk, dv), device=DEV) * 0.1
    s0 = s_sep.clone()
    prev = _window_inputs(B, W, H, dk, dv, torch.bfloat16, 50)[:5]
    nxt = _window_inputs(B, W, H, dk, dv, torch.bfloat16, 51)[:5]
    acc_l = np.random.default_rng(3).integers(0, W + 1, size=B)
    acc = torch.tensor(acc_l, dtype=torch.int32, device=DEV)
    s_fused = s_sep.clone()
    kda.decode_replay(*prev, acc, s_sep)
    o_sep = kda.decode_window(*nxt, s_sep)
    o_fused = kda.decode_replay_window(prev, acc, *nxt, s_fused)
    torch.cuda.synchronize()
    assert torch.equal(o_fused, o_sep) and torch.equal(s_fused, s_sep)
    for b in (0, 17, 39):
        n = int(acc_l[b])
        if n:
            cols = [x[b, :n].cpu() for x in prev]
            _, fin, _ = oracle.recurrent(*cols, [0, n], s0[b:b + 1].cpu())
            assert_close(s_sep[b], fin[0], torch.bfloat16, f"request {b} replayed state")
        o, _, _ = oracle.recurrent(*[x[b].cpu() for x in nxt], [0, W], s_sep[b:b + 1].cpu())
        assert_close(o_sep[b], o, torch.bfloat16, f"request {b} window outputs")
    assert kda.get_device_error() == 0
    bad = acc.clone()
    bad[7] = W + 1
    s_bad = s0.clone()
    kda.decode_replay(*prev, bad, s_bad)
    assert kda.get_device_error() == 5  # KDA_ERR_DEVICE_CHECK
    assert torch.equal(s_bad[7], s0[7])
    s_ref = s0.clone()
    kda.decode_replay(*prev, acc, s_ref)  # the other requests as with a valid length
    torch.cuda.synchronize()
    assert torch.equal(s_bad[8], s_ref[8])
    assert kda.get_device_error() == 0


def test_decode_replay_bad_accept_length_sets_error_and_keeps_state():
    B, W, H = 3, 2, 2
    q, k, v, z, beta, state = _window_inputs(B, W, H, 64, 64, torch.float32, 23)
    before = state.clone()
    kda.decode_replay(q, k, v, z, beta, torch.tensor([1, 3, -1], dtype=torch.int32, device=DEV),
                      state)
    assert kda.get_device_error() == 5  # KDA_ERR_DEVICE_CHECK
    assert torch.equal(state[1], before[1]) and torch.equal(state[2], before[2])
    assert not torch.equal(state[0], before[0])
    assert kda.get_device_error() == 0


# ------------------------------------------------------ state checkpoints ---

def _oracle_checkpoints(p, every):
    """State after every `every` tokens of each sequence: the oracle's final
    state of that prefix (from the sequence's initial state)."""
    cu = p.cu_seqlens_host
    H = p.meta["num_heads"]
    res = []
    for n in range(len(cu) - 1):
        for j in range(1, (cu[n + 1] - cu[n]) // every + 1):
            a, b = cu[n], cu[n] + j * every
            s0 = None if p.initial_state is None else p.initial_state[n:n + 1].cpu()
            _, fin, _ = oracle.recurrent(p.q[a:b].cpu(), p.k[a:b].cpu(), p.v[a:b].cpu(),
                                         p.z[a:b].cpu(), p.beta[a:b].cpu(), [0, b - a], s0)
            res.append(fin[0])
    return np.stack(res) if res else np.zeros((0, H, p.meta["dk"], p.meta["dv"]))


@pytest.mark.parametrize("entry,dtype,dk,dv", [
    ("chunk_fwd", torch.bfloat16, 128, 128),   # tensor-core kernel
    ("chunk_fwd", torch.float32, 64, 32),      # CUDA-core chunked kernel
    ("recurrent_fwd", torch.float32, 32, 64),
    ("chunk_fwd_noalloc", torch.bfloat16, 128, 128),
])
def test_state_checkpoints(entry, dtype, dk, dv):
    lens = [64, 200, 0, 130, 256, 63, 512]
    p = workloads.random_problem(lens, 2, dk, dv, dtype, z_std=1.0, init_std=0.1, seed=13,
                                 device=DEV)
    out, fin, ck = getattr(kda, entry)(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                       cu_seqlens_host=p.cu_seqlens_host, checkpoint_every=64)
    torch.cuda.synchronize()
    assert ck.shape[0] == sum(n // 64 for n in lens) == 18
    ref = _oracle_checkpoints(p, 64)
    assert_close(ck, ref, dtype, "checkpoints")
    # the checkpoint that ends a sequence equals its final state
    offs = kda.checkpoint_offsets(p.cu_seqlens_host, 64)
    assert torch.equal(ck[offs[1] - 1], fin[0])   # sequence 0 has length 64
    assert torch.equal(ck[offs[5] - 1], fin[4])   # sequence 4 has length 256
    assert kda.get_device_error() == 0


def test_state_checkpoints_with_split_sequences():
    """Long sequences split across SMs (workspace): checkpoints come from the
    final pass, which runs every segment from its true entry state."""
    p = workloads.random_problem([3000, 1100], 2, 128, 128, torch.bfloat16, z_mean=-1.0,
                                 init_std=0.1, seed=14, device=DEV)
    assert kda.chunk_fwd_workspace_size(2, 4100, 2, 128, 128, torch.bfloat16,
                                        p.cu_seqlens_host) > 0  # the split is taken
    out, fin, ck = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                 cu_seqlens_host=p.cu_seqlens_host, workspace="auto",
                                 checkpoint_every=256)
    torch.cuda.synchronize()
    assert ck.shape[0] == 3000 // 256 + 1100 // 256
    ref = _oracle_checkpoints(p, 256)
    for i in range(ck.shape[0]):
        assert_close(ck[i], ref[i], torch.bfloat16, f"checkpoint {i}")
    assert kda.get_device_error() == 0


# ------------------------------------------------- full-size workloads -----
#
# Every (sequence, head) of each full workload against the oracle.  The oracle
# runs piece by piece (groups of sequences, or of heads for a single long
# sequence) on all host cores; the whole-tensor relative L2 error, the worst
# per-head value and max|err| / RMS over the whole tensor are accumulated
# across the pieces and checked at the end.

def _full_check(p, results, io_dtype=torch.bfloat16):
    """results: {label: (out, final_state)} of GPU runs on Problem p; each is
    compared with the oracle over every (sequence, head)."""
    H = p.meta["num_heads"]
    cu = p.cu_seqlens_host
    acc = {lab: (WholeTensorError(H, io_dtype), WholeTensorError(H)) for lab in results}
    for (n0, n1), (h0, h1) in problem_pieces(p):
        a, b = cu[n0], cu[n1]
        sl = lambda x: x[a:b, h0:h1].cpu()
        s0 = None if p.initial_state is None else p.initial_state[n0:n1, h0:h1].cpu()
        ro, rf, _ = oracle.recurrent(sl(p.q), sl(p.k), sl(p.v), sl(p.z), sl(p.beta),
                                     [x - a for x in cu[n0:n1 + 1]], s0)
        for lab, (out, fin) in results.items():
            acc[lab][0].add(out[a:b, h0:h1].cpu(), ro, head_axis=1, heads=range(h0, h1))
            acc[lab][1].add(fin[n0:n1, h0:h1].cpu(), rf, head_axis=1, heads=range(h0, h1))
    for lab in results:
        print(acc[lab][0].check(io_dtype, f"{p.name} {lab} out"))
        print(acc[lab][1].check(io_dtype, f"{p.name} {lab} final state"))


def _run_prefill(p, **kw):
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             cu_seqlens_host=p.cu_seqlens_host, **kw)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    return out, fin


def test_full_prefill_workload():
    """4 x 4096 tokens, 16 heads: every output and final state, unsplit and
    with the split across SMs that scratch allows (64 units on 152 SMs)."""
    p = workloads.prefill_workload("prefill", device=DEV)
    res = {"unsplit": _run_prefill(p)}
    if _ws_bytes(p) > 0:
        res["split"] = _run_prefill(p, workspace="auto")
    _full_check(p, res)


@pytest.mark.parametrize("name", ["long", "long_slow"])
def test_full_long_workload(name):
    """One 65536-token sequence, 32 heads, unsplit and split across SMs."""
    p = workloads.prefill_workload(name, device=DEV)
    assert _ws_bytes(p) > 0
    _full_check(p, {"unsplit": _run_prefill(p), "split": _run_prefill(p, workspace="auto")})


def test_full_varlen_workload():
    """The bench step: 64 sequences of 256..8192 tokens, 32 heads, initial
    and final states -- every (sequence, head)."""
    p = workloads.prefill_workload("varlen", device=DEV)
    _full_check(p, {"chunk_fwd": _run_prefill(p)})


def test_full_decode_workload():
    """256 requests x 32 heads, 1000 steps in place: every step's output of
    every (request, head) and every final state against the oracle's
    1000-token recurrence per (request, head)."""
    steps, N, H = 1000, 256, 32
    d = workloads.decode_workload(N, H, 128, 128, steps=steps, device=DEV)
    s0 = d.state.clone()
    outs = torch.empty((steps, N, H, 128), dtype=torch.bfloat16, device=DEV)
    for t in range(steps):
        kda.decode_step(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], d.state, out=outs[t])
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    acc_o, acc_s = WholeTensorError(H, torch.bfloat16), WholeTensorError(H)
    per = 16  # requests per oracle piece (16 x 32 sequences of 1000 tokens)
    for r0 in range(0, N, per):
        r1 = min(N, r0 + per)
        seq = lambda x: x[:, r0:r1].transpose(0, 1).reshape(-1, *x.shape[2:]).cpu()
        cu = [i * steps for i in range(r1 - r0 + 1)]
        ro, rf, _ = oracle.recurrent(seq(d.q), seq(d.k), seq(d.v), seq(d.z), seq(d.beta), cu,
                                     s0[r0:r1].cpu())
        acc_o.add(seq(outs), ro, head_axis=1)
        acc_s.add(d.state[r0:r1].cpu(), rf, head_axis=1)
    print(acc_o.check(torch.bfloat16, "decode 1000 steps out"))
    print(acc_s.check(torch.bfloat16, "decode 1000 steps state"))


def test_tensor_core_fp16_range_check():
    """The tensor-core path's dense products take fp16 operands.  A bf16 v
    beyond the fp16 range (|v| >= 65504, which bf16 holds) is flagged with
    KDA_ERR_DEVICE_CHECK in the device error word, and the next call on the
    same context is correct."""
    p = workloads.random_problem([130, 70], 2, 128, 128, torch.bfloat16, init_std=0.1, seed=31,
                                 device=DEV)
    v_big = p.v.clone()
    v_big[100, 1, 5] = 1.0e5
    assert float(v_big[100, 1, 5]) >= 65504.0
    assert kda.get_device_error() == 0
    kda.chunk_fwd(p.q, p.k, v_big, p.z, p.beta, p.cu_seqlens, p.initial_state,
                  cu_seqlens_host=p.cu_seqlens_host)
    assert kda.get_device_error() == 5  # KDA_ERR_DEVICE_CHECK
    # an initial state beyond the range is flagged as well
    s_big = p.initial_state.clone()
    s_big[0, 0, 3, 3] = 7.0e4
    kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, s_big,
                  cu_seqlens_host=p.cu_seqlens_host)
    assert kda.get_device_error() == 5
    assert kda.get_device_error() == 0  # cleared by the read
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    _check_all(p, out, fin, torch.bfloat16)
    # the fp32 recurrent path takes the same large v without complaint
    o2, f2 = kda.recurrent_fwd(p.q, p.k, v_big, p.z, p.beta, p.cu_seqlens, p.initial_state)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    ro, rf, _ = oracle.recurrent(p.q, p.k, v_big, p.z, p.beta, p.cu_seqlens_host,
                                 p.initial_state)
    assert_close(o2, ro, torch.bfloat16, "recurrent out with |v| = 1e5")


# ------------------------------------------- long sequences split across SMs --

def _ws_bytes(p):
    return kda.chunk_fwd_workspace_size(p.num_seqs, p.total_tokens, p.meta["num_heads"],
                                        p.meta["dk"], p.meta["dv"], p.q.dtype, p.cu_seqlens_host)


@pytest.mark.parametrize("lens,H,init", [([3000], 4, None), ([5000, 1200, 64, 0, 700], 2, 0.1)])
def test_split_matches_unsplit_and_oracle(lens, H, init):
    """With workspace, few long sequences are cut into segments (transition M
    and zero-start state per segment, a prefix scan, then a second pass); the
    result must match the unsplit kernel and the oracle."""
    p = workloads.random_problem(lens, H, 128, 128, torch.bfloat16, init_std=init, seed=21,
                                 device=DEV)
    assert _ws_bytes(p) > 0  # a split is planned for this shape
    o1, f1 = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                           cu_seqlens_host=p.cu_seqlens_host)
    o2, f2 = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                           cu_seqlens_host=p.cu_seqlens_host, workspace="auto")
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert_close(o2, o1, torch.bfloat16, "split vs unsplit out", both_stored=True)
    assert_close(f2, f1, torch.bfloat16, "split vs unsplit final")
    _check_all(p, o2, f2, torch.bfloat16)


def test_split_final_state_may_alias_initial_state():
    p = workloads.random_problem([4000, 900], 3, 128, 128, torch.bfloat16, init_std=0.1, seed=22,
                                 device=DEV)
    s0 = p.initial_state.clone()
    ro, rf, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, s0)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             final_state=p.initial_state, cu_seqlens_host=p.cu_seqlens_host,
                             workspace="auto")
    torch.cuda.synchronize()
    assert_close(out, ro, torch.bfloat16, "out")
    assert_close(fin, rf, torch.bfloat16, "final_state")


def test_expired_device_wait_reports_timeout_and_recovers():
    """A bounded device wait that runs out (made unsatisfiable on purpose by the
    testing hook) ends the kernel with KDA_ERR_TIMEOUT in the error word, no
    trap; the next call on the same context is correct."""
    p = workloads.random_problem([200, 70], 2, 128, 128, torch.bfloat16, init_std=0.1, seed=23,
                                 device=DEV)
    assert kda.get_device_error() == 0
    kda.testing_inject_wait_timeout(1)
    kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                  cu_seqlens_host=p.cu_seqlens_host)
    assert kda.get_device_error() == 4  # KDA_ERR_TIMEOUT
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    _check_all(p, out, fin, torch.bfloat16)


# ----------------------- small states (a CTA per unit, or a warp when many) --

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk", [32, 64])
def test_small_state_path(dtype, dk):
    """dv = 32, dk <= 64 (the CUDA-core path runs a CTA per (sequence, head)
    here): ragged lengths with a long one (many token blocks), checkpoints,
    the gate log-scale, against the oracle."""
    lens = [1, 0, 31, 64, 65, 2000]
    p = workloads.random_problem(lens, 3, dk, 32, dtype, z_mean=-1.0, init_std=0.2, seed=33,
                                 device=DEV)
    A = torch.tensor([0.3, -0.4, 0.9])
    out, fin, ck = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                 cu_seqlens_host=p.cu_seqlens_host, a_log=A.to(DEV),
                                 checkpoint_every=64)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    ro, rf, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host,
                                 p.initial_state, a_log=A)
    assert_close(out, ro, dtype, "out")
    assert_close(fin, rf, dtype, "final_state")
    offs = kda.checkpoint_offsets(p.cu_seqlens_host, 64)
    assert ck.shape[0] == offs[-1] == 1 + 1 + 31
    assert torch.equal(ck[offs[4] - 1], fin[3])  # the 64-token sequence ends on a checkpoint
    # and one gate per head
    zh = p.z[:, :, 0].contiguous()
    out2, fin2 = kda.chunk_fwd(p.q, p.k, p.v, zh, p.beta, p.cu_seqlens, p.initial_state)
    torch.cuda.synchronize()
    zb = zh.cpu()[:, :, None].expand(-1, -1, dk).contiguous()
    ro2, rf2, _ = oracle.recurrent(p.q, p.k, p.v, zb, p.beta, p.cu_seqlens_host, p.initial_state)
    assert_close(out2, ro2, dtype, "per-head gate out")
    assert_close(fin2, rf2, dtype, "per-head gate final_state")


@pytest.mark.parametrize("dtype,dk", [(torch.float32, 32), (torch.bfloat16, 64)])
def test_small_state_inputs_not_16_byte_aligned(dtype, dk):
    """q, k, v, z that start off a 16-byte boundary take the small-state
    path's element-wise staging (aligned inputs are copied in by cp.async):
    the same results bit for bit."""
    p = workloads.random_problem([70, 5, 130], 2, dk, 32, dtype, init_std=0.2, seed=37,
                                 device=DEV)
    o1, f1 = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state)
    mq, mk, mv, mz = (_misaligned(x) for x in (p.q, p.k, p.v, p.z))
    assert all(x.data_ptr() % 16 for x in (mq, mk, mv, mz))
    o2, f2 = kda.chunk_fwd(mq, mk, mv, mz, p.beta, p.cu_seqlens, p.initial_state)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    _check_all(p, o1, f1, dtype)


def test_small_state_many_units():
    """More (sequence, head) units than the small-state path gives a CTA each
    (1,024): 600 sequences x 2 heads run one warp per unit, against the
    oracle."""
    lens = np.random.default_rng(5).integers(0, 40, size=600).tolist()
    p = workloads.random_problem(lens, 2, 32, 32, torch.float32, init_std=0.2, seed=35,
                                 device=DEV)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             cu_seqlens_host=p.cu_seqlens_host)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    _check_all(p, out, fin, torch.float32)


def test_many_short_sequences():
    """More sequences than the tensor-core launcher's longest-first order
    table holds (6144): 7000 sequences of 0..12 tokens, unsplit and with the
    workspace offered, against the oracle."""
    lens = np.random.default_rng(3).integers(0, 13, size=7000).tolist()
    p = workloads.random_problem(lens, 2, 128, 128, torch.bfloat16, init_std=0.1, seed=34,
                                 device=DEV)
    for ws in (None, "auto"):
        out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                                 cu_seqlens_host=p.cu_seqlens_host, workspace=ws)
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        _check_all(p, out, fin, torch.bfloat16)


def test_split_with_a_workspace_smaller_than_the_best_plan():
    """A workspace below what the best split needs: kda_chunk_fwd takes the
    best plan that fits (fewer, longer segments) and stays exact."""
    p = workloads.random_problem([6000, 900], 2, 128, 128, torch.bfloat16, init_std=0.1,
                                 seed=35, device=DEV)
    need = _ws_bytes(p)
    assert need > 0
    small = torch.empty((need // 3) // 256 * 256, dtype=torch.uint8, device=DEV)
    out, fin = kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                             cu_seqlens_host=p.cu_seqlens_host, workspace=small)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    _check_all(p, out, fin, torch.bfloat16)
