"""The chunked-form reverse mode (tests/chunked_backward_form.py), the algebra a
tensor-core backward evaluates, against the oracle's per-token reverse mode,
which tests/test_oracle_backward.py pins to finite differences.  Agreement to
1e-9 relative on every gradient, for several chunk sizes (including chunks
that do not divide the sequence and a chunk of one token), validates each term
of the derivation."""
import numpy as np
import pytest

import oracle
from tests.chunked_backward_form import chunked_backward


def _case(rng, T, D, E, with_state=True, z_scale=1.5):
    q = rng.standard_normal((T, 1, D))
    k = rng.standard_normal((T, 1, D))
    v = rng.standard_normal((T, 1, E))
    z = rng.normal(0, z_scale, size=(T, 1, D))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, 1))))
    s0 = rng.normal(0, 0.3, size=(1, 1, D, E)) if with_state else None
    do = rng.standard_normal((T, 1, E))
    dfin = rng.standard_normal((1, 1, D, E))
    return q, k, v, z, b, s0, do, dfin


@pytest.mark.parametrize("chunk", [1, 4, 7, 16])
@pytest.mark.parametrize("with_state", [True, False])
def test_chunked_reverse_mode_equals_per_token_reverse_mode(chunk, with_state):
    rng = np.random.default_rng(chunk + 10 * with_state)
    T, D, E = 23, 6, 5
    q, k, v, z, b, s0, do, dfin = _case(rng, T, D, E, with_state)
    ref = oracle.backward(q, k, v, z, b, [0, T], s0, do, dfin)
    got = chunked_backward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0],
                           None if s0 is None else s0[0, 0], do[:, 0], dfin[0, 0], chunk=chunk)
    names = ("dq", "dk", "dv", "dz", "dbeta", "d_initial")
    refs = [ref[0][:, 0], ref[1][:, 0], ref[2][:, 0], ref[3][:, 0], ref[4][:, 0], ref[5][0, 0]]
    for name, x, r in zip(names, got, refs):
        err = np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-300)
        assert err <= 1e-9, (name, err)


def test_chunked_reverse_mode_with_gate_scale_and_strong_decay():
    rng = np.random.default_rng(7)
    T, D, E = 19, 4, 4
    q, k, v, z, b, s0, do, dfin = _case(rng, T, D, E, True, z_scale=3.0)
    z += 2.0  # gates near their floor
    ref = oracle.backward(q, k, v, z, b, [0, T], s0, do, dfin, a_log=np.array([0.6]))
    got = chunked_backward(q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], s0[0, 0], do[:, 0],
                           dfin[0, 0], chunk=8, a_log=0.6)
    refs = [ref[0][:, 0], ref[1][:, 0], ref[2][:, 0], ref[3][:, 0], ref[4][:, 0], ref[5][0, 0]]
    for x, r in zip(got, refs):
        assert np.linalg.norm(x - r) <= 1e-9 * np.linalg.norm(r)


@pytest.mark.parametrize("z_mean", [0.0, 6.0, -3.0])
def test_cancellation_free_log_decay_gradient(z_mean):
    """The log-decay gradient the tensor-core kernel sums (only crossing pairs
    of the chunk-internal products, the state terms split at r) equals the
    plain reverse cumulative sum of dG, and the oracle, to 1e-9: slow decay
    (z mean 6), fast decay (z mean -3) and the plain workload spread."""
    rng = np.random.default_rng(31 + int(z_mean))
    T, D, E = 37, 6, 5
    q, k, v, z, b, s0, do, dfin = _case(rng, T, D, E, True)
    z = z + z_mean
    ref = oracle.backward(q, k, v, z, b, [0, T], s0, do, dfin)
    args = (q[:, 0], k[:, 0], v[:, 0], z[:, 0], b[:, 0], s0[0, 0], do[:, 0], dfin[0, 0])
    plain = chunked_backward(*args, chunk=16)
    cross = chunked_backward(*args, chunk=16, dg_form="crossing")
    for x, y in zip(plain, cross):
        assert np.linalg.norm(x - y) <= 1e-12 * max(np.linalg.norm(y), 1e-300)
    assert np.linalg.norm(cross[3] - ref[3][:, 0]) <= 1e-9 * np.linalg.norm(ref[3][:, 0])
