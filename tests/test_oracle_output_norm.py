"""Pins of the oracle's output norm (per-head RMS norm, the reading of the
output norm named in blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构",
section "三条容易被忽略的代价" (1)): a hand-computed row, the closed form of a
constant row, scale invariance, the weight acting per channel, and the mean
square of the result."""
import numpy as np

import oracle


def test_hand_computed_row():
    # o = (3, 4): mean square 12.5, root 3.5355339..., eps 0
    y = oracle.rms_norm(np.array([[3.0, 4.0]]), np.ones((1, 2)), 0.0)
    np.testing.assert_allclose(y, [[3 / 12.5 ** 0.5, 4 / 12.5 ** 0.5]], rtol=1e-15)
    np.testing.assert_allclose(y, [[0.848528137423857, 1.131370849898476]], rtol=1e-14)


def test_constant_row_and_epsilon():
    c, eps = -0.5, 1e-2
    y = oracle.rms_norm(np.full((2, 3, 8), c), np.ones((3, 8)), eps)
    np.testing.assert_allclose(y, c / np.sqrt(c * c + eps), rtol=1e-15)


def test_scale_invariance_weight_and_mean_square():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((5, 4, 32))
    w = rng.standard_normal((4, 32))
    ones = np.ones((4, 32))
    y = oracle.rms_norm(o, ones, 0.0)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * o, ones, 0.0), y, rtol=1e-13)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rms_norm(o, w, 0.0), y * w, rtol=1e-13)
    # heads are normalised separately: scaling one head changes only that head
    o2 = o.copy()
    o2[:, 1] *= 100.0
    y2 = oracle.rms_norm(o2, ones, 1e-6)
    y1 = oracle.rms_norm(o, ones, 1e-6)
    np.testing.assert_allclose(y2[:, [0, 2, 3]], y1[:, [0, 2, 3]], rtol=1e-15)
