"""The tensor-core prefill's chunk algebra, step by step in fp64 numpy (test
infrastructure: tests/test_chunked_forward_form.py checks it against the
oracle's per-token recurrence, which validates the derivation the kernel
implements independently of any GPU rounding).

Per 64-token chunk with four 16-token subtiles (the recurrence of
mhpq.cn/news/56770, section "KDA 到底在算什么", evaluated chunkwise; the lower
bound on the gate keeps a subtile's decay within e^{-80}):
  * r_a = cumulative log-decay before subtile a, G_t inclusive through t.
  * Query side of subtile a: Q~_t = q^_t e^{G_t - r_a}, K~q_t = k^_t e^{G_t - r_a}.
  * Key side for query subtile a: K^(a)_j = k^_j e^{r_a - G_j} for j in subtiles
    0..a, built along the chain K^(a+1) = K^(a) e^{r_{a+1} - r_a}.
  * P[t, j] = Q~_t . K^(a)_j (j <= t), A[t, j] = beta_t K~q_t . K^(a)_j (j < t)
    for t in subtile a: one product of [Q~; K~q] with the packed K^(0..3).
  * T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution, then
    T = (I - N + N^2 - N^3) D^{-1} with D the block diagonal, N = D^{-1} L.
  * T' = T diag(beta), U = T' (V - K+ S), O = Q+ S + P U,
    S <- Diag(e^{G_C}) S + Khat^T U,  Q+ = q^ e^{G}, K+ = k^ e^{G}, Khat = k^ e^{G_C - G}.
"""
import numpy as np

GMIN = -5.0
C, SUB = 64, 16


def _unit(x, eps):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def _block_inverse(A):
    """(I + A)^{-1} for strictly lower A by diagonal solves and the series."""
    n = A.shape[0]
    nb = (n + SUB - 1) // SUB
    Dinv = np.zeros((n, n))
    for b in range(nb):
        s, e = b * SUB, min((b + 1) * SUB, n)
        blk = np.eye(e - s) + A[s:e, s:e]
        X = np.eye(e - s)
        for i in range(e - s):  # forward substitution, one column of the inverse at a time
            for r in range(i + 1, e - s):
                X[r] -= blk[r, i] * X[i]
        Dinv[s:e, s:e] = X
    L = A.copy()
    for b in range(nb):
        s, e = b * SUB, min((b + 1) * SUB, n)
        L[s:e, s:e] = 0.0
    N = Dinv @ L
    series = np.eye(n) - N + N @ N - N @ N @ N  # N^4 = 0 with four blocks
    return series @ Dinv


def chunk_forward(q, k, v, z, beta, s0=None, a_log=0.0, eps=1e-6, slip=None):
    """One sequence, one head: q, k, z [T, dk], v [T, dv], beta [T].
    Returns (out [T, dv], final state [dk, dv]).  `slip` plants one mistake
    (test use only): 'reference_off' (the query side of subtile a > 0 against
    r_{a-1}), 'chain_factor' (K^(a) chained by e^{r_a} instead of
    e^{r_a - r_{a-1}}), 'state_decay' (S carried without Diag(e^{G_C})),
    'key_end' (Khat = k^ e^{-G} instead of k^ e^{G_C - G})."""
    q, k, v, z = (np.asarray(x, dtype=np.float64) for x in (q, k, v, z))
    beta = np.asarray(beta, dtype=np.float64)
    T, D = q.shape
    S = np.zeros((D, v.shape[1])) if s0 is None else np.asarray(s0, dtype=np.float64).copy()
    qh, kh = _unit(q, eps), _unit(k, eps)
    g = GMIN / (1.0 + np.exp(-np.exp(a_log) * z))
    out = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        c1 = min(c0 + C, T)
        n = c1 - c0
        G = np.cumsum(g[c0:c1], axis=0)  # [n, D], inclusive
        nsub = (n + SUB - 1) // SUB
        r = [np.zeros(D)] + [G[a * SUB - 1] for a in range(1, nsub)]  # r_a
        # the packed key side K^(a) for a = 0..nsub-1, rows j = 0 .. 16(a+1)-1, by the chain
        Ka = []
        base = np.zeros((n, D))
        for j in range(min(SUB, n)):  # K^(0): subtile 0 keys at reference r_0 = 0
            base[j] = kh[c0 + j] * np.exp(r[0] - G[j])
        Ka.append(base)
        for a in range(1, nsub):
            chain = r[a] if slip == "chain_factor" else r[a] - r[a - 1]
            prev = Ka[-1] * np.exp(chain)  # chain factor e^{r_a - r_{a-1}} <= 1
            for j in range(a * SUB, min((a + 1) * SUB, n)):  # the new diagonal subtile
                prev[j] = kh[c0 + j] * np.exp(r[a] - G[j])
            Ka.append(prev)
        P = np.zeros((n, n))
        A = np.zeros((n, n))
        for t in range(n):
            a = t // SUB
            ra = r[a - 1] if (slip == "reference_off" and a > 0) else r[a]
            qt = qh[c0 + t] * np.exp(G[t] - ra)
            kq = kh[c0 + t] * np.exp(G[t] - ra)
            for j in range(t + 1):
                P[t, j] = qt @ Ka[a][j]
                if j < t:
                    A[t, j] = beta[c0 + t] * (kq @ Ka[a][j])
        Tp = _block_inverse(A) * beta[None, c0:c1]
        Qp = qh[c0:c1] * np.exp(G)
        Kp = kh[c0:c1] * np.exp(G)
        Kt = kh[c0:c1] * np.exp((0.0 if slip == "key_end" else G[-1]) - G)
        U = Tp @ (v[c0:c1] - Kp @ S)
        out[c0:c1] = Qp @ S + P @ U
        S = (S if slip == "state_decay" else np.exp(G[-1])[:, None] * S) + Kt.T @ U
    return out, S
