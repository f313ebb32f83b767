"""Pins of the oracle's affine segment summary and prefix scan (the
context-parallel scheme of blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构",
section "第二层"): the transition M and offset S~ against the independent
dense-matrix form, the affine identity S_out = M S_in + S~ against the
recurrence, and the scan of per-segment summaries against one pass over the
whole sequence."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.dense_form import dense_states


def _alpha(z):
    return np.exp(-5.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64))))


@pytest.mark.parametrize("T", [1, 3, 7])
def test_summary_equals_dense_products(T):
    """M = A_T ... A_1 and S~ = the state from zeros, both from the dense form
    (A_s = (I - b_s k_s k_s^T) Diag(alpha_s) as explicit matrices)."""
    p = workloads.random_problem([T], 1, 6, 5, torch.float32, seed=40 + T)
    m, st = oracle.affine_summary(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host)
    q, k, v = (x[:, 0].double().numpy() for x in (p.q, p.k, p.v))
    a, b = _alpha(p.z[:, 0].numpy()), p.beta[:, 0].double().numpy()
    _, s_zero = dense_states(q, k, v, a, b, np.zeros((6, 5)), oracle.DEFAULT_EPS)
    _, s_eye = dense_states(q, k, np.zeros((T, 6)), a, b, np.eye(6), oracle.DEFAULT_EPS)
    np.testing.assert_allclose(st[0, 0], s_zero[-1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(m[0, 0], s_eye[-1], rtol=0, atol=1e-12)


def test_affine_identity_against_the_recurrence():
    """For any entering state, the recurrence's final state is M S_in + S~."""
    p = workloads.random_problem([40, 0, 17], 3, 16, 8, torch.float32, init_std=0.7, seed=44)
    m, st = oracle.affine_summary(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host)
    _, fin, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state)
    s_in = p.initial_state.double().numpy()
    np.testing.assert_allclose(np.matmul(m, s_in) + st, fin, rtol=0, atol=1e-12)
    # a zero-length sequence is the identity map with no offset
    np.testing.assert_array_equal(m[1], np.broadcast_to(np.eye(16), (3, 16, 16)))
    np.testing.assert_array_equal(st[1], 0.0)


@pytest.mark.parametrize("cuts", [[0, 37, 80, 130], [0, 64, 64, 130], [0, 1, 129, 130]])
def test_scan_of_segment_summaries_equals_one_pass(cuts):
    """Summaries of consecutive segments, scanned from the initial state, give
    each segment's entering state and, at the end, the whole pass's final state."""
    T = cuts[-1]
    p = workloads.random_problem([T], 2, 16, 12, torch.float32, init_std=0.5, seed=45)
    ms, ss = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sl = lambda x: x[a:b]
        m, st = oracle.affine_summary(sl(p.q), sl(p.k), sl(p.v), sl(p.z), sl(p.beta), [0, b - a])
        ms.append(m)
        ss.append(st)
    ms, ss = np.stack(ms), np.stack(ss)
    for r, a in enumerate(cuts[:-1]):
        entry = oracle.state_scan(ms, ss, p.initial_state, count=r)
        _, ref, _ = oracle.recurrent(p.q[:a], p.k[:a], p.v[:a], p.z[:a], p.beta[:a], [0, a],
                                     p.initial_state)
        np.testing.assert_allclose(entry, ref, rtol=0, atol=1e-11)
    _, fin, _ = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, [0, T], p.initial_state)
    np.testing.assert_allclose(oracle.state_scan(ms, ss, p.initial_state), fin, rtol=0,
                               atol=1e-11)


def test_scan_special_cases():
    rng = np.random.default_rng(3)
    s0 = rng.standard_normal((2, 3, 4, 5))
    m = rng.standard_normal((2, 2, 3, 4, 4))
    s = rng.standard_normal((2, 2, 3, 4, 5))
    np.testing.assert_array_equal(oracle.state_scan(m, s, s0, count=0), s0)
    np.testing.assert_array_equal(oracle.state_scan(m, s, None, count=0), 0.0)
    eye = np.broadcast_to(np.eye(4), m.shape).copy()
    np.testing.assert_allclose(oracle.state_scan(eye, s, s0), s0 + s[0] + s[1], atol=1e-14)
    # the order matters: M_1 (M_0 S + S~_0) + S~_1
    ref = np.matmul(m[1], np.matmul(m[0], s0) + s[0]) + s[1]
    np.testing.assert_allclose(oracle.state_scan(m, s, s0), ref, atol=1e-13)
