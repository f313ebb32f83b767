"""The window kernels' scaled-state algebra (tests/scaled_state_form.py)
against the oracle's per-token recurrence in fp64: the window's outputs are
those of the recurrence run over the replayed prefix and then the drafts,
and the stored state is the recurrence's after the prefix.  Agreement to
1e-10 validates the derivation the kernels implement; each planted slip
fails it, and the renormalisation interval is checked against the fp32
range the kernels hold Gamma^{-1} in."""
import numpy as np
import pytest

import oracle
from tests.scaled_state_form import scaled_state_window


def _inputs(T, D, E, seed, zmean=0.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(zmean, 1.5, size=(T, 1, D))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, 1))))
    s0 = rng.normal(0, 0.3, size=(1, 1, D, E))
    return q, k, v, z, b, s0


def _check(q, k, v, z, b, s0, nrep, a_log=None, slip=None):
    T = q.shape[0]
    ro, _, _ = oracle.recurrent(q, k, v, z, b, [0, T], s0,
                                a_log=None if a_log is None else np.array([a_log]))
    _, rs, _ = oracle.recurrent(q[:nrep], k[:nrep], v[:nrep], z[:nrep], b[:nrep], [0, nrep], s0,
                                a_log=None if a_log is None else np.array([a_log]))
    o, s, _ = scaled_state_window(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], s0[0, 0], nrep,
                                  a_log=a_log, slip=slip)
    err_o = np.linalg.norm(o - ro[nrep:, 0]) / max(np.linalg.norm(ro[nrep:, 0]), 1e-300)
    err_s = np.linalg.norm(s - rs[0, 0]) / np.linalg.norm(rs[0, 0])
    return err_o if T > nrep else 0.0, err_s


@pytest.mark.parametrize("nrep,W", [(0, 1), (0, 4), (1, 4), (2, 4), (4, 4), (4, 0), (3, 9),
                                    (9, 3), (17, 20), (8, 8)])
def test_scaled_state_equals_recurrence(nrep, W):
    q, k, v, z, b, s0 = _inputs(nrep + W, 8, 6, 300 + 7 * nrep + W)
    err_o, err_s = _check(q, k, v, z, b, s0, nrep)
    assert err_o <= 1e-10 and err_s <= 1e-10


def test_scaled_state_gates_at_their_floor_and_gate_scale():
    q, k, v, z, b, s0 = _inputs(27, 8, 4, 11, zmean=6.0)
    err_o, err_s = _check(q, k, v, z, b, s0, 10, a_log=0.4)
    assert err_o <= 1e-10 and err_s <= 1e-10


@pytest.mark.parametrize("slip", ["gamma_prev", "no_output_term", "update_gamma"])
def test_planted_slips_fail(slip):
    q, k, v, z, b, s0 = _inputs(14, 8, 6, 5)
    err_o, err_s = _check(q, k, v, z, b, s0, 5, slip=slip)
    assert max(err_o, err_s) > 1e-3


def test_renormalisation_keeps_gamma_inverse_in_fp32_range():
    """Every decay at its floor e^-5 (z large): renormalising every 8 tokens
    keeps Gamma^{-1} at most e^40, while one 20-token part without it needs
    e^100, past the largest fp32 value (about e^88.7).  Without the reset the
    algebra is still exact in fp64 -- the interval is a range device."""
    T, D, E = 20, 4, 3
    rng = np.random.default_rng(2)
    q = rng.standard_normal((T, D))
    k = rng.standard_normal((T, D))
    v = rng.standard_normal((T, E))
    z = np.full((T, D), 60.0)
    b = np.full(T, 0.5)
    s0 = rng.normal(0, 0.3, size=(D, E))
    fp32_max = float(np.finfo(np.float32).max)
    _, _, inv8 = scaled_state_window(q, k, v, z, b, s0, 0)
    assert inv8 <= np.exp(40.0) * (1 + 1e-12) and inv8 < fp32_max
    _, _, inv_all = scaled_state_window(q, k, v, z, b, s0, 0, slip="no_renorm")
    assert inv_all > fp32_max
