"""The decode-side calls with the short convolution and the output norm
fused in (kda_decode_step_fused, kda_decode_replay_window_fused), against
the oracle composition of the same steps: oracle.short_conv on the raw q and
k of each request's token stream (from its convolution state), the fp64
recurrence, then oracle.rms_norm of the outputs.  The convolution states the
kernels leave behind are the last raw inputs, compared bit for bit."""
import numpy as np
import pytest
import torch

import linear_attention_layer_gb300 as kda
import oracle
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.load()
    torch.cuda.set_device(0)


def _tokens(shape_bt, H, dk, dv, dtype, g):
    """Raw (pre-convolution) q, k ~ N(0, 1), v, z, beta for [*shape_bt] tokens."""
    f32 = dict(dtype=torch.float32, device=DEV, generator=g)
    q = torch.randn((*shape_bt, H, dk), **f32).to(dtype)
    k = torch.randn((*shape_bt, H, dk), **f32).to(dtype)
    v = torch.randn((*shape_bt, H, dv), **f32).to(dtype)
    z = torch.randn((*shape_bt, H, dk), **f32)
    beta = torch.sigmoid(torch.randn((*shape_bt, H), **f32))
    return q, k, v, z, beta


def _fusion_tensors(B, H, dk, dv, W, g, norm):
    f32 = dict(dtype=torch.float32, device=DEV, generator=g)
    fz = {}
    if W:
        fz["conv_weight_q"] = torch.randn((H, dk, W), **f32) * 0.6
        fz["conv_weight_k"] = torch.randn((H, dk, W), **f32) * 0.6
        if W > 1:
            fz["conv_state_q"] = torch.randn((B, H, dk, W - 1), **f32)
            fz["conv_state_k"] = torch.randn((B, H, dk, W - 1), **f32)
    if norm:
        fz["out_norm_weight"] = 1.0 + 0.3 * torch.randn((H, dv), **f32)
        fz["out_norm_eps"] = EPS
    return fz


def _oracle_stream(q, k, v, z, beta, s0, fz, W, cq0, ck0):
    """One request's token stream [T, H, .] from state s0 [H, dk, dv] and
    convolution states cq0 / ck0 [H, dk, W-1]: (outputs, state, conv states)."""
    T = q.shape[0]
    cu = [0, T]
    if W:
        qy, cq = oracle.short_conv(q, fz["conv_weight_q"], cu, None if cq0 is None else cq0[None])
        ky, ck = oracle.short_conv(k, fz["conv_weight_k"], cu, None if ck0 is None else ck0[None])
    else:
        qy, ky, cq, ck = q, k, None, None
    out, fin, _ = oracle.recurrent(qy, ky, v, z, beta, cu, s0[None])
    if "out_norm_weight" in fz:
        out = oracle.rms_norm(out, fz["out_norm_weight"], EPS)
    return out, fin[0], (None if cq is None else cq[0]), (None if ck is None else ck[0])


@pytest.mark.parametrize("W,norm", [(4, True), (2, False), (1, True), (0, True), (3, True)])
@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 32)])
def test_decode_step_fused_matches_oracle(W, norm, dtype, dk, dv):
    g = torch.Generator(device=DEV).manual_seed(60 + W)
    B, H, steps = 5, 3, 4
    toks = _tokens((steps, B), H, dk, dv, dtype, g)
    state = torch.randn((B, H, dk, dv), device=DEV, generator=g) * 0.1
    fz = _fusion_tensors(B, H, dk, dv, W, g, norm)
    s0 = state.clone()
    c0 = {key: fz[key].clone() for key in ("conv_state_q", "conv_state_k") if key in fz}
    outs = [kda.decode_step_fused(*(x[t] for x in toks), state, **fz) for t in range(steps)]
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    fz_cpu = {kk: vv.cpu() for kk, vv in fz.items() if torch.is_tensor(vv)}
    for b in range(B):
        seq = [x[:, b].cpu() for x in toks]
        ro, rs, rcq, rck = _oracle_stream(*seq, s0[b].cpu(), fz_cpu, W,
                                          c0["conv_state_q"][b].cpu() if W > 1 else None,
                                          c0["conv_state_k"][b].cpu() if W > 1 else None)
        assert_close(torch.stack([o[b] for o in outs]), ro, dtype, f"request {b} outputs")
        assert_close(state[b], rs, dtype, f"request {b} state")
        if W > 1:
            assert torch.equal(fz["conv_state_q"][b].cpu(), torch.from_numpy(rcq).float())
            assert torch.equal(fz["conv_state_k"][b].cpu(), torch.from_numpy(rck).float())


def test_decode_step_fused_without_options_equals_decode_step():
    g = torch.Generator(device=DEV).manual_seed(70)
    q, k, v, z, beta = _tokens((6,), 4, 128, 128, torch.bfloat16, g)
    s1 = torch.randn((6, 4, 128, 128), device=DEV, generator=g) * 0.1
    s2 = s1.clone()
    o1 = kda.decode_step(q, k, v, z, beta, s1)
    o2 = kda.decode_step_fused(q, k, v, z, beta, s2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_fused_draft_verify_replay_loop():
    """Three rounds: each step replays the previous window's accepted prefix
    (raw inputs) and returns the new window's normalised outputs, one kernel
    per step.  Outputs against the oracle composition over the committed
    tokens plus the window's drafts; final states and convolution states
    against the oracle over the accepted tokens only."""
    g = torch.Generator(device=DEV).manual_seed(71)
    B, H, dk, dv, Wc, Wd = 4, 2, 128, 128, 4, 3
    state = torch.randn((B, H, dk, dv), device=DEV, generator=g) * 0.1
    fz = _fusion_tensors(B, H, dk, dv, Wc, g, True)
    s0, cq0, ck0 = state.clone(), fz["conv_state_q"].clone(), fz["conv_state_k"].clone()
    fz_cpu = {kk: vv.cpu() for kk, vv in fz.items() if torch.is_tensor(vv)}
    committed = [[] for _ in range(B)]
    rng = np.random.default_rng(4)
    prev, acc = None, None
    for r in range(4):
        win = _tokens((B, Wd), H, dk, dv, torch.bfloat16, g) if r < 3 else None
        out = kda.decode_replay_window_fused(prev, acc, win, state, **fz)
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        if prev is not None:
            for b in range(B):
                committed[b] += [tuple(x[b, i].cpu() for x in prev) for i in range(int(acc[b]))]
        if win is not None:
            for b in range(B):
                toks = committed[b] + [tuple(x[b, i].cpu() for x in win) for i in range(Wd)]
                seq = [torch.stack([t[j] for t in toks]) for j in range(5)]
                ro, _, _, _ = _oracle_stream(*seq, s0[b].cpu(), fz_cpu, Wc, cq0[b].cpu(),
                                             ck0[b].cpu())
                assert_close(out[b], ro[len(committed[b]):], torch.bfloat16,
                             f"round {r} request {b} window outputs")
        prev = win
        acc = torch.tensor(rng.integers(0, Wd + 1, size=B), dtype=torch.int32, device=DEV)
    for b in range(B):
        n = len(committed[b])
        if n == 0:
            assert torch.equal(state[b], s0[b]) and torch.equal(fz["conv_state_q"][b], cq0[b])
            continue
        seq = [torch.stack([t[j] for t in committed[b]]) for j in range(5)]
        _, rs, rcq, rck = _oracle_stream(*seq, s0[b].cpu(), fz_cpu, Wc, cq0[b].cpu(), ck0[b].cpu())
        assert_close(state[b], rs, torch.bfloat16, f"request {b} state after {n} tokens")
        assert torch.equal(fz["conv_state_q"][b].cpu(), torch.from_numpy(rcq).float())
        assert torch.equal(fz["conv_state_k"][b].cpu(), torch.from_numpy(rck).float())


def test_fused_bad_accept_length_keeps_both_states():
    g = torch.Generator(device=DEV).manual_seed(72)
    B, H, dk, dv, Wd = 3, 2, 64, 64, 2
    state = torch.randn((B, H, dk, dv), device=DEV, generator=g) * 0.1
    fz = _fusion_tensors(B, H, dk, dv, 4, g, True)
    before = (state.clone(), fz["conv_state_q"].clone(), fz["conv_state_k"].clone())
    prev = _tokens((B, Wd), H, dk, dv, torch.float32, g)
    acc = torch.tensor([1, Wd + 1, 0], dtype=torch.int32, device=DEV)
    kda.decode_replay_window_fused(prev, acc, None, state, **fz)
    assert kda.get_device_error() == 5  # KDA_ERR_DEVICE_CHECK
    assert torch.equal(state[1], before[0][1]) and torch.equal(fz["conv_state_q"][1], before[1][1])
    assert torch.equal(state[2], before[0][2]) and torch.equal(fz["conv_state_k"][2], before[2][2])
    assert not torch.equal(state[0], before[0][0])
    assert kda.get_device_error() == 0


def test_fused_decode_gate_log_scale_and_per_head_gate():
    """The fused decode step honours the gate log-scale A and one gate per
    head, like the plain decode step."""
    g = torch.Generator(device=DEV).manual_seed(73)
    B, H, dk, dv, steps = 4, 3, 128, 128, 3
    toks = _tokens((steps, B), H, dk, dv, torch.bfloat16, g)
    A = torch.tensor([0.4, -0.6, 1.1], device=DEV)
    for per_head in (False, True):
        state = torch.randn((B, H, dk, dv), device=DEV, generator=g) * 0.1
        fz = _fusion_tensors(B, H, dk, dv, 4, g, True)
        s0, cq0, ck0 = state.clone(), fz["conv_state_q"].clone(), fz["conv_state_k"].clone()
        zs = toks[3][..., 0].contiguous() if per_head else toks[3]
        outs = [kda.decode_step_fused(toks[0][t], toks[1][t], toks[2][t], zs[t], toks[4][t], state,
                                      a_log=A, **fz) for t in range(steps)]
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        fz_cpu = {kk: vv.cpu() for kk, vv in fz.items() if torch.is_tensor(vv)}
        for b in range(B):
            zb = zs[:, b].cpu()
            if per_head:
                zb = zb[:, :, None].expand(-1, -1, dk).contiguous()
            T = steps
            qy, _ = oracle.short_conv(toks[0][:, b].cpu(), fz_cpu["conv_weight_q"], [0, T], cq0[b:b + 1].cpu())
            ky, _ = oracle.short_conv(toks[1][:, b].cpu(), fz_cpu["conv_weight_k"], [0, T], ck0[b:b + 1].cpu())
            ro, rf, _ = oracle.recurrent(qy, ky, toks[2][:, b].cpu(), zb, toks[4][:, b].cpu(), [0, T],
                                         s0[b:b + 1].cpu(), a_log=A.cpu())
            ro = oracle.rms_norm(ro, fz_cpu["out_norm_weight"], EPS)
            assert_close(torch.stack([o[b] for o in outs]), ro, torch.bfloat16, f"b={b} out")
            assert_close(state[b], rf[0], torch.bfloat16, f"b={b} state")
