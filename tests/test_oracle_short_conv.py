"""Pins for the oracle's short causal convolution + Swish (CPU only).

The page (mhpq.cn/news/56770, the Q/K preprocessing paragraph of section
"KDA 到底在算什么") fixes a causal convolution over the last few positions
followed by Swish; the checks below pin the oracle to facts that do not come
from its own code: the Swish closed form, np.convolve per channel, pure shifts,
linearity before the activation, and that carrying the state across a split
sequence equals one pass."""
import numpy as np

import oracle


def test_swish_closed_form():
    u = np.array([-30.0, -2.0, -0.5, 0.0, 0.5, 2.0, 30.0])
    expect = np.array([-30.0 / (1 + np.exp(30.0)), -2.0 / (1 + np.exp(2.0)),
                       -0.5 / (1 + np.exp(0.5)), 0.0, 0.5 / (1 + np.exp(-0.5)),
                       2.0 / (1 + np.exp(-2.0)), 30.0 / (1 + np.exp(-30.0))])
    assert np.allclose(oracle.swish(u), expect, rtol=1e-15, atol=0)
    # swish(u) - swish(-u) = u (sigmoid(u) + sigmoid(-u) = 1)
    assert np.allclose(oracle.swish(u) - oracle.swish(-u), u, rtol=1e-14, atol=1e-14)


def test_matches_numpy_convolve_per_channel():
    rng = np.random.default_rng(0)
    T, H, D, W = 23, 2, 3, 4
    x = rng.standard_normal((T, H, D))
    w = rng.standard_normal((H, D, W))
    y, fin = oracle.short_conv(x, w, [0, T], activation=False)
    for h in range(H):
        for d in range(D):
            # causal: y[t] = sum_j w[j] x[t - (W-1) + j] = (x * reversed(w))[t]
            full = np.convolve(x[:, h, d], w[h, d, ::-1])
            assert np.allclose(y[:, h, d], full[:T], rtol=1e-13, atol=1e-13)
            assert np.array_equal(fin[0, h, d], x[T - (W - 1):, h, d])


def test_pure_shifts_read_the_state():
    rng = np.random.default_rng(1)
    T, H, D, W = 6, 1, 2, 4
    x = rng.standard_normal((T, H, D))
    st = rng.standard_normal((1, H, D, W - 1))
    ident = np.zeros((H, D, W)); ident[..., W - 1] = 1.0
    y, _ = oracle.short_conv(x, ident, [0, T], st, activation=False)
    assert np.array_equal(y, x)
    oldest = np.zeros((H, D, W)); oldest[..., 0] = 1.0
    y, _ = oracle.short_conv(x, oldest, [0, T], st, activation=False)
    ext = np.concatenate([np.transpose(st[0], (2, 0, 1)), x])  # [state..., x...]
    assert np.array_equal(y, ext[:T])  # y[t] = x[t - 3], the state for t < 3


def test_linearity_before_activation_and_swish_after():
    rng = np.random.default_rng(2)
    T, H, D, W = 9, 2, 2, 3
    x1, x2 = rng.standard_normal((2, T, H, D))
    w = rng.standard_normal((H, D, W))
    lin = lambda x: oracle.short_conv(x, w, [0, 4, T], activation=False)[0]
    assert np.allclose(lin(2.0 * x1 - 0.5 * x2), 2.0 * lin(x1) - 0.5 * lin(x2), atol=1e-13)
    y, _ = oracle.short_conv(x1, w, [0, 4, T])
    assert np.allclose(y, oracle.swish(lin(x1)), rtol=0, atol=0)


def test_state_carried_across_a_split_equals_one_pass():
    rng = np.random.default_rng(3)
    T, H, D, W = 13, 2, 3, 4
    x = rng.standard_normal((T, H, D))
    w = rng.standard_normal((H, D, W))
    s0 = rng.standard_normal((1, H, D, W - 1))
    y, fin = oracle.short_conv(x, w, [0, T], s0)
    for cut in (1, 2, 5):  # pieces shorter and longer than W - 1
        ya, sa = oracle.short_conv(x[:cut], w, [0, cut], s0)
        yb, sb = oracle.short_conv(x[cut:], w, [0, T - cut], sa)
        assert np.allclose(np.concatenate([ya, yb]), y, rtol=1e-14, atol=1e-14)
        assert np.array_equal(sb, fin)


def test_sequences_do_not_see_each_other_and_empty_keeps_state():
    rng = np.random.default_rng(4)
    H, D, W = 1, 2, 4
    x = rng.standard_normal((7, H, D))
    w = rng.standard_normal((H, D, W))
    st = rng.standard_normal((3, H, D, W - 1))
    y, fin = oracle.short_conv(x, w, [0, 2, 2, 7], st)
    y0, _ = oracle.short_conv(x[:2], w, [0, 2], st[0:1])
    y2, _ = oracle.short_conv(x[2:], w, [0, 5], st[2:3])
    assert np.array_equal(y, np.concatenate([y0, y2]))
    assert np.array_equal(fin[1], st[1])  # zero-length sequence: state unchanged
    # a 2-token sequence (shorter than W - 1) keeps the newest state entry
    assert np.array_equal(fin[0, ..., 0], st[0, ..., 2])
    assert np.array_equal(fin[0, ..., 1:], np.transpose(x[:2], (1, 2, 0)))
