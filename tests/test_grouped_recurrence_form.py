"""The small-state kernel's four-tokens-a-pass algebra
(tests/grouped_recurrence_form.py) against the oracle's per-token recurrence
in fp64.  Agreement to 1e-10 validates the derivation the kernel implements;
a plausible slip (a decay ratio off by one token, a missing correction term,
o read before the update instead of after) fails it."""
import numpy as np
import pytest

import oracle
from tests.grouped_recurrence_form import grouped_forward


@pytest.mark.parametrize("T", [1, 3, 4, 5, 8, 63, 64, 65, 130])
def test_grouped_algebra_equals_recurrence(T):
    rng = np.random.default_rng(100 + T)
    D, E = 8, 6
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(0, 1.5, size=(T, 1, D))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, 1))))
    s0 = rng.normal(0, 0.3, size=(1, 1, D, E))
    ro, rf, _ = oracle.recurrent(q, k, v, z, b, [0, T], s0)
    o, f = grouped_forward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], s0[0, 0])
    assert np.linalg.norm(o - ro[:, 0]) <= 1e-10 * np.linalg.norm(ro)
    assert np.linalg.norm(f - rf[0, 0]) <= 1e-10 * np.linalg.norm(rf)


def test_grouped_algebra_gates_at_their_floor_and_gate_scale():
    rng = np.random.default_rng(7)
    T, D, E = 37, 8, 4
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(6.0, 1.0, size=(T, 1, D))
    b = np.ones((T, 1))
    ro, rf, _ = oracle.recurrent(q, k, v, z, b, [0, T], None, a_log=np.array([0.4]))
    o, f = grouped_forward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], None,
                           a_log=np.array(0.4))
    assert np.linalg.norm(o - ro[:, 0]) <= 1e-10 * np.linalg.norm(ro)
    assert np.linalg.norm(f - rf[0, 0]) <= 1e-10 * np.linalg.norm(rf)


@pytest.mark.parametrize("slip", ["ratio_off_by_one", "no_output_term", "end_decay"])
def test_planted_slips_fail(slip):
    rng = np.random.default_rng(21)
    T, D, E = 23, 8, 6
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(0, 1.5, size=(T, 1, D))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, 1))))
    s0 = rng.normal(0, 0.3, size=(1, 1, D, E))
    ro, rf, _ = oracle.recurrent(q, k, v, z, b, [0, T], s0)
    o, f = grouped_forward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], s0[0, 0], slip=slip)
    err = max(np.linalg.norm(o - ro[:, 0]) / np.linalg.norm(ro),
              np.linalg.norm(f - rf[0, 0]) / np.linalg.norm(rf))
    assert err > 3e-3
