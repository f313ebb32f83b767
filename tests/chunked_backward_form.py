"""The chunked (WY / UT) form of KDA and its reverse mode, written out by hand
in fp64 numpy, one chunk at a time: the algebra a tensor-core backward kernel
evaluates.  Test infrastructure: tests/test_chunked_backward_form.py checks it
against the oracle's per-token reverse mode (itself pinned by finite
differences), which validates the derivation before any kernel uses it.

Forward of one chunk of C tokens (mhpq.cn/news/56770, section "KDA 到底在算什么",
evaluated chunkwise; G the inclusive cumulative log-decay per channel, S the
entering state [dk, dv]):
    Q+ = q^ e^{G},  K+ = k^ e^{G},  K- = k^ e^{-G},  K~ = k^ e^{G_C - G}
    A = diag(beta) strict_lower(K+ K-^T),  P = lower(Q+ K-^T)
    T = (I + A)^{-1},  T' = T diag(beta),  R = V - K+ S,  U = T' R
    O = Q+ S + P U,  S' = Diag(e^{G_C}) S + K~^T U
Reverse, given dO and dS' (the gradient w.r.t. the leaving state):
    dU = P^T dO + K~ dS',  dP = lower(dO U^T),  dQ+ = dO S^T,  dK~ = U dS'^T
    dS = Q+^T dO + Diag(e^{G_C}) dS' - K+^T dR,  dR = T'^T dU,  dV = dR,  dK+ = -dR S^T
    dT' = dU R^T,  dT = dT' diag(beta),  dbeta_j += (T^T dT')_jj
    dA = strict_lower(-T^T dT T^T),  dbeta_t += sum_j strict_lower(K+ K-^T)_tj dA_tj
    dK+ += diag(beta) dA K-,  dK- = (diag(beta) dA)^T K+ + dP^T Q+,  dQ+ += dP K-
    then through the exponentials: dG += dQ+ Q+ + dK+ K+ - dK- K- - dK~ K~ (elementwise),
    dG_C += sum_t dK~ K~ + rowsum(S dS') e^{G_C}, and dg = the reverse cumulative sum of dG.
The gate and L2-norm chains per token are those of the per-token reverse mode.
"""
import numpy as np

GMIN = -5.0


def _unit(x, eps):
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    return x * r, r


def chunked_backward(q, k, v, z, beta, s0, d_out, d_fin, chunk=8, a_log=0.0, eps=1e-6,
                     dg_form="plain"):
    """One sequence, one head.  q, k, z: [T, dk]; v, d_out: [T, dv]; beta: [T];
    s0, d_fin: [dk, dv] (None for zeros).  Returns (dq, dk, dv, dz, dbeta, ds0).
    dg_form "crossing": the gradient of the log-decay summed without cancelling
    terms (see _chunk_backward), the form the tensor-core kernel evaluates."""
    q, k, v, z = (np.asarray(x, dtype=np.float64) for x in (q, k, v, z))
    beta = np.asarray(beta, dtype=np.float64)
    d_out = np.asarray(d_out, dtype=np.float64)
    T, D = q.shape
    E = v.shape[1]
    S0 = np.zeros((D, E)) if s0 is None else np.asarray(s0, dtype=np.float64)
    dS = np.zeros((D, E)) if d_fin is None else np.asarray(d_fin, dtype=np.float64).copy()
    qh, rq = _unit(q, eps)
    kh, rk = _unit(k, eps)
    s = np.exp(a_log)
    sig = 1.0 / (1.0 + np.exp(-s * z))
    g = GMIN * sig                                      # log-decay per (token, channel)
    # forward over the chunks: the state entering each one
    starts = list(range(0, T, chunk))
    entering = []
    S = S0.copy()
    for c0 in starts:
        c1 = min(c0 + chunk, T)
        entering.append(S.copy())
        S = _chunk_forward(qh[c0:c1], kh[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1], S)[1]
    dqh, dkh = np.zeros((T, D)), np.zeros((T, D))
    dv, dg, dbeta = np.zeros((T, E)), np.zeros((T, D)), np.zeros(T)
    for ci in range(len(starts) - 1, -1, -1):
        c0 = starts[ci]
        c1 = min(c0 + chunk, T)
        grads = _chunk_backward(qh[c0:c1], kh[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1],
                                entering[ci], d_out[c0:c1], dS, dg_form)
        dqh[c0:c1], dkh[c0:c1], dv[c0:c1], dg[c0:c1], dbeta[c0:c1], dS = grads
    # gate: g = GMIN sigmoid(s z)  ->  dg/dz = GMIN s sigmoid (1 - sigmoid)
    dz = dg * GMIN * s * sig * (1.0 - sig)
    # L2 norm: x^ = x r  ->  dx = r (dx^ - x^ (x^ . dx^))
    dq = rq * (dqh - qh * np.sum(qh * dqh, axis=1, keepdims=True))
    dk = rk * (dkh - kh * np.sum(kh * dkh, axis=1, keepdims=True))
    return dq, dk, dv, dz, dbeta, dS


def _operands(qh, kh, g):
    G = np.cumsum(g, axis=0)
    eG, eC = np.exp(G), np.exp(G[-1])
    return G, qh * eG, kh * eG, kh * np.exp(-G), kh * (eC / eG), eC


def _chunk_forward(qh, kh, v, g, beta, S):
    C = qh.shape[0]
    _, Qp, Kp, Km, Kt, eC = _operands(qh, kh, g)
    L = np.tril(np.ones((C, C)), -1)
    A = beta[:, None] * (L * (Kp @ Km.T))
    P = np.tril(Qp @ Km.T)
    Tp = np.linalg.inv(np.eye(C) + A) * beta[None, :]
    U = Tp @ (v - Kp @ S)
    return Qp @ S + P @ U, eC[:, None] * S + Kt.T @ U


def _chunk_backward(qh, kh, v, g, beta, S, dO, dS1, dg_form="plain"):
    C = qh.shape[0]
    _, Qp, Kp, Km, Kt, eC = _operands(qh, kh, g)
    Ls = np.tril(np.ones((C, C)), -1)
    Li = np.tril(np.ones((C, C)))
    Araw = Kp @ Km.T
    A = beta[:, None] * (Ls * Araw)
    P = Li * (Qp @ Km.T)
    Tm = np.linalg.inv(np.eye(C) + A)
    Tp = Tm * beta[None, :]
    R = v - Kp @ S
    U = Tp @ R
    # products
    dU = P.T @ dO + Kt @ dS1
    dP = Li * (dO @ U.T)
    dQp = dO @ S.T
    dKt = U @ dS1.T
    dS = Qp.T @ dO + eC[:, None] * dS1
    deC = np.sum(S * dS1, axis=1)
    dR = Tp.T @ dU
    dv = dR
    dKp = -dR @ S.T
    dS -= Kp.T @ dR
    # the UT transform
    dTp = dU @ R.T
    dbeta = np.sum(Tm * dTp, axis=0)                 # from T' = T diag(beta)
    dT = dTp * beta[None, :]
    dA = Ls * (-(Tm.T @ dT @ Tm.T))
    dbeta += np.sum(Ls * Araw * dA, axis=1)          # from A = diag(beta) strict_lower(.)
    dAr = beta[:, None] * dA
    dKp += dAr @ Km
    dKm = dAr.T @ Kp + dP.T @ Qp
    dQp += dP @ Km
    # through the exponentials of G
    dqh = dQp * np.exp(np.cumsum(g, axis=0))
    G = np.cumsum(g, axis=0)
    eG = np.exp(G)
    dkh = dKp * eG + dKm * np.exp(-G) + dKt * (eC / eG)
    dG = dQp * Qp + dKp * Kp - dKm * Km - dKt * Kt
    dG[-1] += np.sum(dKt * Kt, axis=0) + deC * eC
    dg = np.cumsum(dG[::-1], axis=0)[::-1]           # G = cumsum(g)
    if dg_form == "crossing":
        # The same sum without the terms that cancel in it: the state parts of
        # dQ+ o Q+ and dK+ o K+ from row r on, the K~ parts before row r, and
        # only those (t, s) pairs of the chunk-internal products with
        # t >= r > s, plus rowsum(S o dS') e^{G_C}:
        #   dg_r = e^{G_C} rowsum(S o dS') + sum_{t>=r} a_t + sum_{t<r} b_t
        #          + sum_{t>=r>s} (dP_ts Q+_t + dAr_ts K+_t) K-_s
        a = (dO @ S.T) * Qp - (dR @ S.T) * Kp
        b = dKt * Kt
        M = (dP[:, :, None] * Qp[:, None, :] + dAr[:, :, None] * Kp[:, None, :]) * Km[None, :, :]
        dg = np.zeros_like(dG)
        for r in range(C):
            dg[r] = deC * eC + a[r:].sum(0) + b[:r].sum(0) + M[r:, :r].sum((0, 1))
    return dqh, dkh, dv, dg, dbeta, dS
