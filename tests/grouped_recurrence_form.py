"""The small-state kernel's four-tokens-a-pass algebra, step by step in fp64
numpy (test infrastructure: tests/test_grouped_recurrence_form.py checks it
against the oracle's per-token recurrence, which validates the derivation the
kernel implements independently of any GPU rounding).

The recurrence of mhpq.cn/news/56770, section "KDA 到底在算什么", taken four
tokens at a time.  For a group j = 0..3 entered with state S, with A_j the
running product of the decays over the group's tokens 0..j (per key row) and
x_i = beta_i e_i:
  * K_j = S^T (A_j k_j),  Q_j = S^T (A_j q_j)     (one pass over S)
  * c_ji = k_j . (A_j / A_i) k_i,  d_ji = q_j . (A_j / A_i) k_i   (i < j)
  * e_j = v_j - K_j - sum_{i<j} c_ji x_i            (a 4 x 4 triangular solve)
  * o_j = Q_j + sum_{i<j} d_ji x_i + (q_j . k_j) x_j
  * S' = A_3 S + sum_i (A_3 / A_i) k_i x_i^T         (one pass over S)
Rows past the sequence's end are k = q = v = 0, decay 1, beta 0.
"""
import numpy as np

GMIN = -5.0


def _unit(x, eps):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def grouped_forward(q, k, v, z, beta, s0, a_log=None, eps=1e-6, group=4, slip=None):
    """q, k, z [T, D], v [T, E], beta [T], s0 [D, E] (or None).  Returns
    (o [T, E], final state [D, E]).  `slip` plants one mistake (test use
    only): 'ratio_off_by_one' (A_j / A_i taken over tokens i..j), 'no_output_term'
    (o_j without (q_j . k_j) x_j), 'end_decay' (S' = A_2 S instead of A_3 S)."""
    T, D = q.shape
    E = v.shape[1]
    scale = np.exp(a_log) if a_log is not None else 1.0
    qh, kh = _unit(q, eps), _unit(k, eps)
    alpha = np.exp(GMIN / (1.0 + np.exp(-scale * z)))
    S = np.zeros((D, E)) if s0 is None else np.array(s0, dtype=np.float64)
    o = np.zeros((T, E))
    for t0 in range(0, T, group):
        n = min(group, T - t0)
        K = np.zeros((group, D))
        Qr = np.zeros((group, D))
        al = np.ones((group, D))
        V = np.zeros((group, E))
        b = np.zeros(group)
        K[:n], Qr[:n], al[:n], V[:n], b[:n] = kh[t0:t0 + n], qh[t0:t0 + n], alpha[t0:t0 + n], \
            v[t0:t0 + n], beta[t0:t0 + n]
        A = np.cumprod(al, axis=0)  # A_j over the group's tokens 0..j

        def rho(j, i):  # A_j / A_i as the product of the decays in between
            lo = i if slip == "ratio_off_by_one" else i + 1
            return np.prod(al[lo:j + 1], axis=0)

        Kj = (A * K) @ S  # [group, E]
        Qj = (A * Qr) @ S
        x = np.zeros((group, E))
        for j in range(group):
            e = V[j] - Kj[j]
            for i in range(j):
                e = e - np.dot(K[j] * rho(j, i), K[i]) * x[i]
            x[j] = b[j] * e
        for j in range(n):
            oj = Qj[j] + (0.0 if slip == "no_output_term" else np.dot(Qr[j], K[j])) * x[j]
            for i in range(j):
                oj = oj + np.dot(Qr[j] * rho(j, i), K[i]) * x[i]
            o[t0 + j] = oj
        last = group - 1
        S = A[last - 1 if slip == "end_decay" else last][:, None] * S
        for i in range(group):
            S = S + np.outer(rho(last, i) * K[i], x[i])
    return o, S
