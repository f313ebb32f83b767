"""The tensor-core prefill's chunk algebra (tests/chunked_forward_form.py:
subtile references, the chained packed key side, the block-diagonal-plus-series
inverse, U = T'(V - K+ S)) against the oracle's per-token recurrence in fp64.
Agreement to 1e-10 validates the derivation the kernel implements; a plausible
slip (a reference off by a subtile, a wrong chain factor, a missing series
term) fails it."""
import numpy as np
import pytest

import oracle
from tests.chunked_forward_form import chunk_forward


@pytest.mark.parametrize("T", [1, 15, 16, 17, 64, 65, 150])
def test_chunk_algebra_equals_recurrence(T):
    rng = np.random.default_rng(T)
    D, E = 8, 6
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(0, 1.5, size=(T, 1, D))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, 1))))
    s0 = rng.normal(0, 0.3, size=(1, 1, D, E))
    ro, rf, _ = oracle.recurrent(q, k, v, z, b, [0, T], s0)
    o, f = chunk_forward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], s0[0, 0])
    assert np.linalg.norm(o - ro[:, 0]) <= 1e-10 * np.linalg.norm(ro)
    assert np.linalg.norm(f - rf[0, 0]) <= 1e-10 * np.linalg.norm(rf)


def test_chunk_algebra_near_the_decay_bound_and_gate_scale():
    """Gates near their floor (a subtile decays by almost e^-80) and a per-head
    scale: the references keep every factor in range."""
    rng = np.random.default_rng(3)
    T, D, E = 128, 8, 8
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(6.0, 1.0, size=(T, 1, D))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, 1))))
    ro, rf, _ = oracle.recurrent(q, k, v, z, b, [0, T], None, a_log=np.array([0.4]))
    o, f = chunk_forward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], None, a_log=0.4)
    assert np.linalg.norm(o - ro[:, 0]) <= 1e-10 * np.linalg.norm(ro)
    assert np.linalg.norm(f - rf[0, 0]) <= 1e-10 * np.linalg.norm(rf)


def test_chunk_algebra_slow_decay_needs_every_series_term():
    """Near-unit retention: tokens three subtiles apart still interact, so the
    last term of the inverse's series (N^3) matters."""
    rng = np.random.default_rng(4)
    T, D, E = 64, 4, 4
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(-7.0, 0.5, size=(T, 1, D))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, 1))))
    ro, rf, _ = oracle.recurrent(q, k, v, z, b, [0, T], None)
    o, f = chunk_forward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], None)
    assert np.linalg.norm(o - ro[:, 0]) <= 1e-10 * np.linalg.norm(ro)
    assert np.linalg.norm(f - rf[0, 0]) <= 1e-10 * np.linalg.norm(rf)


@pytest.mark.parametrize("slip", ["reference_off", "chain_factor", "state_decay", "key_end"])
def test_planted_slips_fail(slip):
    rng = np.random.default_rng(41)
    T, D, E = 150, 8, 6
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(-2.0, 1.5, size=(T, 1, D))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, 1))))
    s0 = rng.normal(0, 0.3, size=(1, 1, D, E))
    ro, rf, _ = oracle.recurrent(q, k, v, z, b, [0, T], s0)
    o, f = chunk_forward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], s0[0, 0], slip=slip)
    err = max(np.linalg.norm(o - ro[:, 0]) / np.linalg.norm(ro),
              np.linalg.norm(f - rf[0, 0]) / np.linalg.norm(rf))
    assert err > 1e-3
