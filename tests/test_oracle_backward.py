"""Pins for the oracle's backward pass (CPU only).

The backward is the reverse mode of the per-token recurrence of
mhpq.cn/news/56770, section "KDA 到底在算什么", with the gate of
blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构", section "下界衰减".
The pages print no gradient, so every check here compares it with central
finite differences of the forward oracle in fp64: for a loss
L = sum(dO * out) + sum(dS * final_state) with random dO, dS, the gradient
with respect to each input element must equal (L(x + h) - L(x - h)) / 2h.
A dropped term, a sign or a transposed operand in any step of the reverse
pass shows up as an O(1) relative error on some input.
"""
import numpy as np
import pytest

import oracle


def _problem(rng, lens, H, dk, dv, with_state=True):
    T = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    z = rng.normal(0, 1.5, size=(T, H, dk))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    s0 = rng.normal(0, 0.3, size=(len(lens), H, dk, dv)) if with_state else None
    return cu, [q, k, v, z, b, s0]


def _check(cu, args, d_out, d_fin, a_log=None, samples=None, rng=None, tol=1e-7):
    def loss(xs):
        o, f, _ = oracle.recurrent(*xs[:5], cu, xs[5], a_log=a_log)
        return float((o * d_out).sum() + ((f * d_fin).sum() if d_fin is not None else 0.0))

    grads = oracle.backward(*args[:5], cu, args[5], d_out, d_fin, a_log=a_log)
    for i, x in enumerate(args):
        if x is None:
            continue
        idxs = list(np.ndindex(x.shape))
        if samples is not None and len(idxs) > samples:
            idxs = [idxs[j] for j in rng.choice(len(idxs), samples, replace=False)]
        h = 1e-6
        scale = max(np.abs(grads[i]).max(), 1e-3)
        for idx in idxs:
            xp = [a.copy() if a is not None else None for a in args]
            xm = [a.copy() if a is not None else None for a in args]
            xp[i][idx] += h
            xm[i][idx] -= h
            fd = (loss(xp) - loss(xm)) / (2 * h)
            assert abs(fd - grads[i][idx]) <= tol * scale, (i, idx, fd, grads[i][idx])
    return grads


def test_backward_matches_finite_differences_small():
    rng = np.random.default_rng(0)
    cu, args = _problem(rng, [2, 3], 2, 3, 2)
    d_out = rng.standard_normal((5, 2, 2))
    d_fin = rng.standard_normal((2, 2, 3, 2))
    _check(cu, args, d_out, d_fin)


def test_backward_with_gate_log_scale_and_zero_length_sequence():
    rng = np.random.default_rng(1)
    cu, args = _problem(rng, [3, 0, 4], 2, 4, 3)
    d_out = rng.standard_normal((7, 2, 3))
    d_fin = rng.standard_normal((3, 2, 4, 3))
    g = _check(cu, args, d_out, d_fin, a_log=np.array([0.5, -1.1]))
    # a zero-length sequence passes the state's gradient straight through
    assert np.array_equal(g[5][1], d_fin[1])


def test_backward_across_stored_state_blocks():
    """150 tokens: the states are rebuilt from blocks of 64, so a token on each
    side of the block boundaries and the final partial block are sampled."""
    rng = np.random.default_rng(2)
    cu, args = _problem(rng, [150], 1, 3, 2)
    d_out = rng.standard_normal((150, 1, 2))
    d_fin = rng.standard_normal((1, 1, 3, 2))
    _check(cu, args, d_out, d_fin, samples=24, rng=rng)


def test_backward_without_initial_or_final_state_gradient():
    rng = np.random.default_rng(3)
    cu, args = _problem(rng, [4], 1, 3, 3, with_state=False)
    d_out = rng.standard_normal((4, 1, 3))
    grads = _check(cu, args, d_out, None)
    # with no initial state its gradient is still returned (state = 0)
    assert grads[5].shape == (1, 1, 3, 3) and np.isfinite(grads[5]).all()
