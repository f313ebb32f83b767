"""fp64 oracle of the Q/K preprocessing convolution (TEST INFRASTRUCTURE:
imported only by ``tests/`` and ``bench.py``'s CPU legs, through ``oracle``).

mhpq.cn/news/56770, section "KDA 到底在算什么" (the Q/K preprocessing
paragraph): query and key first go through a short causal convolution that
looks only at the most recent few positions, then a Swish activation, then the
L2 normalisation.  The page gives neither the width nor the form; the reading
taken here is a depthwise (one filter per head and channel) causal
convolution of width W with no bias,

    y[t, h, d] = swish( sum_{j=0}^{W-1} w[h, d, j] * x[t - (W - 1) + j, h, d] ),
    swish(u) = u * sigmoid(u),

where positions before a sequence's first token read the sequence's
convolution state (its W - 1 inputs before the start, oldest first; zeros
when none is given).  The state after the sequence is its last W - 1 inputs,
continued from the incoming state when the sequence is shorter than W - 1.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def swish(u):
    """u * sigmoid(u), written as u / (1 + e^-u)."""
    u = np.asarray(u, dtype=np.float64)
    return u / (1.0 + np.exp(-u))


def short_conv(x, weight, cu_seqlens, conv_state=None, *, activation=True):
    """x [T, H, D], weight [H, D, W], cu_seqlens [N + 1], conv_state
    [N, H, D, W - 1] or None.  Returns (y [T, H, D], final_state
    [N, H, D, W - 1]) in float64.  ``activation=False`` returns the
    convolution before the Swish."""
    x, w = _f64(x), _f64(weight)
    cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    T, H, D = x.shape
    W = w.shape[-1]
    N = len(cu) - 1
    st = np.zeros((N, H, D, W - 1)) if conv_state is None else _f64(conv_state).copy()
    y = np.zeros((T, H, D))
    fin = np.zeros((N, H, D, W - 1))
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        # the sequence's inputs preceded by its state: ext[(W - 1) + i] = x[a + i]
        ext = np.concatenate([np.transpose(st[n], (2, 0, 1)), x[a:b]], axis=0)
        for i in range(b - a):
            acc = np.zeros((H, D))
            for j in range(W):
                acc += w[:, :, j] * ext[i + j]
            y[a + i] = acc
        fin[n] = np.transpose(ext[ext.shape[0] - (W - 1):], (1, 2, 0)) if W > 1 else fin[n]
    return (swish(y) if activation else y), fin
