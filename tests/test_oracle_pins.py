"""Pins for the fp64 oracle (CPU only, no GPU).

Each test checks the oracle against something other than itself: values the
pages print, closed forms of the recurrence, a hand-derived fixture, and an
independent dense-matrix formulation.  The mistakes each one is meant to catch
are named in its docstring.

Sources: the state update and read-out of mhpq.cn/news/56770, section
"KDA 到底在算什么"; the gate and the 16-token bound of blog.higcp.com
"猜想：K3 可能是最适合 TPU 的 MoE 架构", section "下界衰减".
"""
import math

import numpy as np
import pytest

import oracle
from tests.dense_form import dense_states, unit


def _run1(q, k, v, g_or_z, beta, S0=None, raw=True, eps=0.0):
    """One sequence, one head: add the [T, H=1, d] axes and call the oracle."""
    T = q.shape[0]
    out, fin, _ = oracle.recurrent(
        q[:, None, :], k[:, None, :], v[:, None, :], g_or_z[:, None, :],
        beta[:, None], np.array([0, T]),
        None if S0 is None else S0[None, None], raw_log_decay=raw, eps=eps)
    return out[:, 0, :], fin[0, 0]


def _orthonormal(rng, n, d):
    m, _ = np.linalg.qr(rng.standard_normal((d, d)))
    return m[:, :n].T.copy()  # n orthonormal rows


# ---------------------------------------------------------------- gate ----

def test_gate_special_values(fixture_reader):
    """g = gmin*sigmoid(z): sigmoid(0)=1/2 gives gmin/2; saturation gives gmin;
    z -> -inf gives 0; printed alpha_min = e^gmin ~ 6.7e-3.  Catches a wrong
    sign, a wrong gmin, a missing sigmoid or exp(+z) in place of exp(-z)."""
    fx = fixture_reader("gate_bounds.txt")
    gmin = fx["gmin"][0]
    assert oracle.log_decay(np.array([0.0]))[0] == gmin / 2
    assert oracle.log_decay(np.array([60.0]))[0] == gmin
    assert abs(oracle.log_decay(np.array([-60.0]))[0]) < 1e-25
    # sigmoid(ln 3) = 3/4 exactly in real arithmetic
    assert abs(oracle.log_decay(np.array([math.log(3.0)]))[0] - 0.75 * gmin) < 1e-15
    z = np.linspace(-8, 8, 101)
    g = oracle.log_decay(z)
    assert np.all(np.diff(g) < 0) and np.all(g < 0) and np.all(g > gmin)
    alpha_min = math.exp(gmin)
    digits = int(fx["alpha_min_printed_digits"][0])
    assert float(f"{alpha_min:.{digits - 1}e}") == fx["alpha_min_printed"][0]


def test_tile_bound_never_crossed(fixture_reader):
    """North-star check (5): the cumulative log-decay over any 16-token tile
    stays in (-80, 0], with -80 reached only when sigmoid saturates to 1."""
    fx = fixture_reader("gate_bounds.txt")
    tile = int(fx["tile_tokens"][0])
    lo = fx["tile_log_decay_lower"][0]
    rng = np.random.default_rng(0)
    for mu, sd in [(0.0, 1.0), (0.0, 1.5), (2.0, 1.0), (-2.0, 1.0), (8.0, 1.0)]:
        z = rng.normal(mu, sd, size=(tile * 64, 8))
        g = oracle.log_decay(z)
        for s in range(0, z.shape[0] - tile + 1, 7):  # every start offset class
            tot = g[s:s + tile].sum(axis=0)
            assert np.all(tot > lo) and np.all(tot < 0)
    # saturated: equals the bound, does not cross it
    g = oracle.log_decay(np.full((tile, 4), 80.0))
    assert np.all(g.sum(axis=0) >= lo)
    # the reciprocal bound e^80 fits bf16's range (max ~3.39e38)
    import torch
    assert math.exp(-lo) < float(torch.finfo(torch.bfloat16).max)


def test_l2norm_special_values():
    """Pythagorean triples normalise exactly (eps = 0); a zero vector stays zero
    with the library eps; eps enters under the square root."""
    out = oracle.l2norm(np.array([[3.0, 4.0, 12.0], [0.0, 0.0, 0.0]]), eps=0.0)
    assert np.allclose(out[0], [3 / 13, 4 / 13, 12 / 13], atol=1e-16, rtol=0)
    out = oracle.l2norm(np.array([[0.0, 0.0, 0.0], [0.0, 1.0, 0.0]]), eps=1e-6)
    assert np.all(out[0] == 0.0)
    assert abs(out[1, 1] - 1.0 / math.sqrt(1.0 + 1e-6)) < 1e-16


# ------------------------------------------------------------ recurrence --

def test_hand_derived_three_tokens(fixture_reader):
    """Three tokens worked by hand (fixture): pins decay-before-erase, row-wise
    decay, read-out after the update and the final state."""
    fx = fixture_reader("hand_dk2_dv2_t3.txt")
    r = lambda key, shape: np.array(fx[key]).reshape(shape)
    out, fin = _run1(r("q", (3, 2)), r("k", (3, 2)), r("v", (3, 2)), r("g", (3, 2)),
                     r("beta", (3,)), r("initial_state", (2, 2)), raw=True, eps=0.0)
    assert np.allclose(out, r("out", (3, 2)), atol=1e-14, rtol=0)
    assert np.allclose(fin, r("final_state", (2, 2)), atol=1e-14, rtol=0)


def test_orthonormal_keys_recall_exactly():
    """North-star check (1): orthonormal keys, beta=1, alpha=1; querying a past
    key returns its value exactly.  Keys and queries are scaled (not unit) so a
    missing L2-normalisation fails."""
    rng = np.random.default_rng(1)
    dk, dv, n = 16, 12, 10
    keys = _orthonormal(rng, n, dk)
    vals = rng.standard_normal((n, dv))
    scale = rng.uniform(0.5, 3.0, size=(n, 1))
    q = np.concatenate([rng.standard_normal((n, dk)), keys[::-1] * 2.5])
    k = np.concatenate([keys * scale, rng.standard_normal((n, dk))])
    v = np.concatenate([vals, rng.standard_normal((n, dv))])
    beta = np.concatenate([np.ones(n), np.zeros(n)])
    g = np.zeros((2 * n, dk))
    out, fin = _run1(q, k, v, g, beta, None, raw=True, eps=0.0)
    assert np.allclose(out[n:], vals[::-1], atol=1e-12, rtol=0)
    assert np.allclose(fin, keys.T @ vals, atol=1e-12, rtol=0)


def test_rewrite_same_key_keeps_latest():
    """North-star check (2): two beta=1 writes to one key keep only the latest
    value along that key; the part of S0 orthogonal to it is untouched."""
    rng = np.random.default_rng(2)
    dk, dv = 8, 6
    kk = rng.standard_normal(dk)
    kh = kk / np.linalg.norm(kk)
    S0 = rng.standard_normal((dk, dv))
    v1, v2 = rng.standard_normal(dv), rng.standard_normal(dv)
    # the second write uses -2k: same line, opposite sign, different scale
    q = np.stack([kk, -3 * kk])
    k = np.stack([kk, -2 * kk])
    v = np.stack([v1, v2])
    out, fin = _run1(q, k, v, np.zeros((2, dk)), np.ones(2), S0, raw=True, eps=0.0)
    assert np.allclose(out[1], v2, atol=1e-12)
    assert np.allclose(fin.T @ (-kh), v2, atol=1e-12)
    P = np.eye(dk) - np.outer(kh, kh)
    assert np.allclose(fin, P @ S0 - np.outer(kh, v2), atol=1e-12)


def test_beta_zero_decays_rows_by_product_of_alpha():
    """North-star check (3): after one write, beta=0 leaves S_T = Diag(prod
    alpha) S_1, row by row (dk != dv, so a column-wise decay fails)."""
    rng = np.random.default_rng(3)
    dk, dv, T = 6, 4, 9
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    g = -rng.uniform(0, 5, size=(T, dk))
    beta = np.zeros(T)
    beta[0] = 1.0
    _, S1 = _run1(q[:1], k[:1], v[:1], g[:1], beta[:1], None, raw=True, eps=0.0)
    _, ST = _run1(q, k, v, g, beta, None, raw=True, eps=0.0)
    decay = np.exp(g[1:].sum(axis=0))
    assert np.allclose(ST, decay[:, None] * S1, rtol=1e-13, atol=0)
    # through the gate itself: z = 0 gives alpha = e^{-2.5} every token
    _, STz = _run1(q, k, v, np.zeros((T, dk)), beta, None, raw=False, eps=0.0)
    _, S1z = _run1(q[:1], k[:1], v[:1], np.zeros((1, dk)), beta[:1], None, raw=False, eps=0.0)
    assert np.allclose(STz, math.exp(-2.5 * (T - 1)) * S1z, rtol=1e-13, atol=0)


def test_gate_log_scale_per_head():
    """The gate's per-head log-scale A (blog.higcp.com "下界衰减": g = g_min
    sigmoid(e^A z)): two heads with different A against the independent dense
    form with alpha built here from e^{A_h} z.  Catches A applied to g instead
    of z, A used without the exponential, the wrong head's A, or A ignored."""
    rng = np.random.default_rng(21)
    T, dk, dv = 6, 5, 3
    A = np.array([0.7, -1.3])
    q = rng.standard_normal((T, 2, dk))
    k = rng.standard_normal((T, 2, dk))
    v = rng.standard_normal((T, 2, dv))
    z = rng.normal(0, 1.5, size=(T, 2, dk))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, 2))))
    S0 = rng.normal(0, 0.5, size=(1, 2, dk, dv))
    eps = 1e-6
    out, fin, _ = oracle.recurrent(q, k, v, z, beta, np.array([0, T]), S0, eps=eps, a_log=A)
    for h in range(2):
        alpha = np.exp(-5.0 / (1.0 + np.exp(-math.exp(A[h]) * z[:, h])))
        outs, states = dense_states(q[:, h], k[:, h], v[:, h], alpha, beta[:, h], S0[0, h], eps)
        assert np.max(np.abs(out[:, h] - outs)) < 1e-12
        assert np.max(np.abs(fin[0, h] - states[-1])) < 1e-12
    # beta = 0 after one write: rows decay by prod alpha with alpha = e^{-5 sigmoid(e^A z)}
    b0 = np.zeros((T, 2))
    b0[0] = 1.0
    _, f1, _ = oracle.recurrent(q[:1], k[:1], v[:1], z[:1], b0[:1], np.array([0, 1]), None,
                                eps=0.0, a_log=A)
    _, fT, _ = oracle.recurrent(q, k, v, z, b0, np.array([0, T]), None, eps=0.0, a_log=A)
    for h in range(2):
        g = -5.0 / (1.0 + np.exp(-math.exp(A[h]) * z[1:, h]))
        assert np.allclose(fT[0, h], np.exp(g.sum(axis=0))[:, None] * f1[0, h], rtol=1e-13,
                           atol=0)


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_dense_product_form(T):
    """North-star check (4): the explicit sum of dense matrix products agrees
    with the oracle to 1e-12, for every output and the final state."""
    rng = np.random.default_rng(10 + T)
    dk, dv = 7, 5
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    z = rng.normal(0, 1.5, size=(T, dk))
    beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
    S0 = rng.normal(0, 0.5, size=(dk, dv))
    eps = 1e-6
    alpha = np.exp(-5.0 / (1.0 + np.exp(-z)))
    outs, states = dense_states(q, k, v, alpha, beta, S0, eps)
    out, fin = _run1(q, k, v, z, beta, S0, raw=False, eps=eps)
    assert np.max(np.abs(out - outs)) < 1e-12
    assert np.max(np.abs(fin - states[-1])) < 1e-12


def test_dense_form_packed_varlen_multihead():
    """Packed batch: 3 sequences (lengths 3, 0, 4), 2 heads, nonzero initial
    states.  Each (sequence, head) must match its own dense evaluation, so a
    wrong head stride, sequence offset or state index fails."""
    rng = np.random.default_rng(20)
    lens = [3, 0, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, dk, dv, eps = int(cu[-1]), 2, 5, 3, 1e-6
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    z = rng.standard_normal((T, H, dk))
    beta = rng.uniform(0, 1, size=(T, H))
    S0 = rng.standard_normal((3, H, dk, dv))
    out, fin, _ = oracle.recurrent(q, k, v, z, beta, cu, S0, eps=eps)
    alpha = np.exp(-5.0 / (1.0 + np.exp(-z)))
    for n in range(3):
        a, b = cu[n], cu[n + 1]
        for h in range(H):
            if b == a:
                assert np.array_equal(fin[n, h], S0[n, h])
                continue
            outs, states = dense_states(q[a:b, h], k[a:b, h], v[a:b, h], alpha[a:b, h],
                                        beta[a:b, h], S0[n, h], eps)
            assert np.max(np.abs(out[a:b, h] - outs)) < 1e-12
            assert np.max(np.abs(fin[n, h] - states[-1])) < 1e-12


# -------------------------------------------------------------- invariants --

def _rand_problem(rng, T, H, dk, dv):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    z = rng.normal(0, 1.5, size=(T, H, dk))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, z, beta


def test_beta_one_write_then_read_returns_value():
    """With beta_t = 1 the new state maps the unit key k_t to v_t for any
    previous state and any decay: S_t^T k_t = v_t."""
    rng = np.random.default_rng(30)
    T, dk, dv = 6, 8, 8
    q, k, v, z, beta = _rand_problem(rng, T, 1, dk, dv)
    beta[-1] = 1.0
    q[-1] = 4.0 * k[-1]  # read along the key just written
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, fin, _ = oracle.recurrent(q, k, v, z, beta, [0, T], S0, eps=0.0)
    kh = unit(k[-1, 0], 0.0)
    assert np.allclose(fin[0, 0].T @ kh, v[-1, 0], atol=1e-12)
    assert np.allclose(out[-1, 0], v[-1, 0], atol=1e-12)


def test_contraction_bound_per_token():
    """(I - b k k^T) Diag(a) has spectral norm <= 1 for b in [0,1], a in (0,1],
    |k| = 1, so ||S_t||_F <= ||S_{t-1}||_F + b_t ||v_t||.  Checked by chaining
    single-token decode steps (which also pins decode_step == recurrent)."""
    rng = np.random.default_rng(31)
    T, H, dk, dv = 20, 2, 6, 5
    q, k, v, z, beta = _rand_problem(rng, T, H, dk, dv)
    S = rng.standard_normal((1, H, dk, dv)) * 3
    full_out, full_fin, _ = oracle.recurrent(q, k, v, z, beta, [0, T], S)
    for t in range(T):
        o, S_new = oracle.decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], z[t:t + 1],
                                      beta[t:t + 1], S)
        for h in range(H):
            lhs = np.linalg.norm(S_new[0, h])
            rhs = np.linalg.norm(S[0, h]) + beta[t, h] * np.linalg.norm(v[t, h])
            assert lhs <= rhs + 1e-12
        assert np.allclose(o[0], full_out[t], atol=1e-12)
        S = S_new
    assert np.allclose(S, full_fin, atol=1e-12)


def test_linearity_in_state_and_values():
    """The update is linear in (S_0, V) jointly: outputs and final state of
    a*(S0, V) + b*(S0', V') equal a*result + b*result'."""
    rng = np.random.default_rng(32)
    T, H, dk, dv = 12, 2, 6, 4
    q, k, v1, z, beta = _rand_problem(rng, T, H, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    s1 = rng.standard_normal((1, H, dk, dv))
    s2 = rng.standard_normal((1, H, dk, dv))
    a, b = 0.7, -1.3
    o1, f1, _ = oracle.recurrent(q, k, v1, z, beta, [0, T], s1)
    o2, f2, _ = oracle.recurrent(q, k, v2, z, beta, [0, T], s2)
    o3, f3, _ = oracle.recurrent(q, k, a * v1 + b * v2, z, beta, [0, T], a * s1 + b * s2)
    assert np.allclose(o3, a * o1 + b * o2, atol=1e-12)
    assert np.allclose(f3, a * f1 + b * f2, atol=1e-12)


def test_value_columns_evolve_independently():
    """Each dv column of S evolves on its own: running a subset of value
    columns gives that subset of the full result (what dv-slicing relies on)."""
    rng = np.random.default_rng(33)
    T, H, dk, dv = 10, 1, 6, 8
    q, k, v, z, beta = _rand_problem(rng, T, H, dk, dv)
    s0 = rng.standard_normal((1, H, dk, dv))
    o, f, _ = oracle.recurrent(q, k, v, z, beta, [0, T], s0)
    cols = [1, 4, 5]
    os_, fs, _ = oracle.recurrent(q, k, v[..., cols], z, beta, [0, T], s0[..., cols])
    assert np.allclose(os_, o[..., cols], atol=1e-13)
    assert np.allclose(fs, f[..., cols], atol=1e-13)


@pytest.mark.parametrize("split", [0, 1, 7, 15])
def test_split_prefix_invariance(split):
    """The final state of tokens [0, t) fed as the initial state of [t, T)
    reproduces the whole run (prefix reuse / context-parallel carry)."""
    rng = np.random.default_rng(34)
    T, H, dk, dv = 15, 2, 5, 4
    q, k, v, z, beta = _rand_problem(rng, T, H, dk, dv)
    s0 = rng.standard_normal((1, H, dk, dv))
    o, f, _ = oracle.recurrent(q, k, v, z, beta, [0, T], s0)
    oa, fa, _ = oracle.recurrent(q[:split], k[:split], v[:split], z[:split], beta[:split],
                                 [0, split], s0)
    ob, fb, _ = oracle.recurrent(q[split:], k[split:], v[split:], z[split:], beta[split:],
                                 [0, T - split], fa)
    assert np.allclose(np.concatenate([oa, ob]), o, atol=1e-12)
    assert np.allclose(fb, f, atol=1e-12)


def test_scalar_decay_is_gated_deltanet():
    """With one retention for all channels (scalar alpha) KDA reduces to the
    Gated DeltaNet update S_t = alpha_t (I - b k k^T) S_{t-1} + b k v^T (the
    scalar commutes with the erase); with alpha = 1 it is plain DeltaNet."""
    rng = np.random.default_rng(35)
    T, dk, dv = 9, 6, 5
    q, k, v, _, beta = _rand_problem(rng, T, 1, dk, dv)
    a = rng.uniform(0.2, 1.0, size=T)
    for alpha in (a, np.ones(T)):
        g = np.repeat(np.log(alpha)[:, None, None], dk, axis=2)
        S0 = rng.standard_normal((dk, dv))
        out, fin, _ = oracle.recurrent(q, k, v, g, beta, [0, T], S0[None, None],
                                       raw_log_decay=True, eps=0.0)
        S = S0.copy()
        for t in range(T):
            kh = unit(k[t, 0], 0.0)
            qh = unit(q[t, 0], 0.0)
            S = alpha[t] * (S - beta[t, 0] * np.outer(kh, kh @ S)) + beta[t, 0] * np.outer(kh, v[t, 0])
            assert np.allclose(out[t, 0], S.T @ qh, atol=1e-12)
        assert np.allclose(fin[0, 0], S, atol=1e-12)


def test_zero_length_sequences_pass_state_through():
    """A zero-length sequence returns its initial state unchanged."""
    rng = np.random.default_rng(36)
    s0 = rng.standard_normal((2, 1, 3, 3))
    q = np.zeros((0, 1, 3))
    out, fin, _ = oracle.recurrent(q, q, q, q, np.zeros((0, 1)), [0, 0, 0], s0)
    assert out.shape == (0, 1, 3)
    assert np.array_equal(fin, s0)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(37)
    T, H, dk, dv = 40, 6, 8, 8
    q, k, v, z, beta = _rand_problem(rng, T, H, dk, dv)
    cu = [0, 13, 13, 40]
    o1, f1, n1 = oracle.recurrent(q, k, v, z, beta, cu, threads=1)
    o4, f4, n4 = oracle.recurrent(q, k, v, z, beta, cu, threads=4)
    assert n1 == 1 and n4 >= 1
    assert np.array_equal(o1, o4) and np.array_equal(f1, f4)
