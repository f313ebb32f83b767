"""Independent dense-matrix formulation of the KDA recurrence, for pinning the oracle.

The state update of mhpq.cn/news/56770, section "KDA 到底在算什么",
S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T, is affine in S.
Unrolled from S_0 it is the explicit sum of matrix products

    S_t = (A_t ... A_1) S_0 + sum_{j<=t} (A_t ... A_{j+1}) b_j k_j v_j^T,
    A_s = (I - b_s k_s k_s^T) Diag(a_s),

which this module builds with dense numpy matmuls (dk x dk transition
matrices), never forming the rank-one update the oracle uses.  Only for tiny T.
"""
import numpy as np


def unit(x, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def dense_states(q, k, v, alpha, beta, S0, eps):
    """Single sequence, single head.  q,k: [T,dk]; v: [T,dv]; alpha: [T,dk];
    beta: [T]; S0: [dk,dv].  Returns (outs [T,dv], states [T,dk,dv])."""
    q = unit(q, eps)
    k = unit(k, eps)
    T, dk = k.shape
    A = [(np.eye(dk) - beta[s] * np.outer(k[s], k[s])) @ np.diag(alpha[s]) for s in range(T)]
    outs, states = [], []
    for t in range(T):
        prod = np.eye(dk)
        for s in range(t, -1, -1):  # A_t ... A_0
            prod = prod @ A[s]
        S = prod @ S0
        for j in range(t + 1):
            P = np.eye(dk)
            for s in range(t, j, -1):  # A_t ... A_{j+1}
                P = P @ A[s]
            S = S + P @ (beta[j] * np.outer(k[j], v[j]))
        states.append(S)
        outs.append(S.T @ q[t])
    return np.array(outs), np.array(states)
