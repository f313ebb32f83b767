"""The window kernels' scaled-state algebra, token by token in fp64 numpy
(test infrastructure: tests/test_scaled_state_form.py checks it against the
oracle's per-token recurrence, which validates the derivation the kernels
implement independently of any GPU rounding).

The recurrence of mhpq.cn/news/56770, section "KDA 到底在算什么", with the
state held as S~ = Gamma^{-1} S, Gamma = Diag of the decays' running product
since the part (the replayed prefix, the window of drafts) began or was last
renormalised.  For token t with raw q, k, r_q = 1 / sqrt(|q|^2 + eps),
r_k likewise, decays alpha_t and Gamma_t = Gamma_{t-1} alpha_t:
  * Sbar_t = Diag(alpha_t) S_{t-1} = Gamma_t S~, so
    Sbar_t^T k^ = r_k S~^T (Gamma_t k) and Sbar_t^T q^ = r_q S~^T (Gamma_t q)
  * e_t = v_t - Sbar_t^T k^
  * o_t = Sbar_t^T q^ + beta_t (k^ . q^) e_t     (S_t^T q^, read after the write)
  * S~ += (Gamma_t^{-1} k) (beta_t r_k e_t)^T     (S_t = Gamma_t S~)
  * S = Gamma_t S~ and Gamma = I where the next token starts a part, every
    `renorm` tokens of a part, and where the replayed state is stored.
The decay never enters as its own pass over the state: one token costs
three multiply-adds per state element (two sums, one update).
"""
import numpy as np

GMIN = -5.0


def scaled_state_window(q, k, v, z, beta, s0, nrep, a_log=None, eps=1e-6, renorm=8,
                        slip=None):
    """q, k, z [T, D], v [T, E], beta [T], s0 [D, E]; tokens [0, nrep) are the
    replayed prefix, [nrep, T) the window.  Returns (o [T - nrep, E] the
    window's outputs, the state after the replayed prefix [D, E], the largest
    entry of Gamma^{-1} met).  `slip` plants one mistake (test use only):
    'gamma_prev' (products with Gamma_{t-1}), 'no_output_term' (o without
    beta (k^ . q^) e), 'update_gamma' (the update with Gamma k instead of
    Gamma^{-1} k), 'no_renorm' (Gamma never reset)."""
    T, D = q.shape
    E = v.shape[1]
    scale = np.exp(a_log) if a_log is not None else 1.0
    alpha = np.exp(GMIN / (1.0 + np.exp(-scale * z)))
    St = np.array(s0, dtype=np.float64)  # S~ (Gamma = I at the start)
    stored = St.copy() if nrep == 0 else None
    outs = []
    gam = np.ones(D)
    inv_max = 1.0

    def fresh(j):
        if slip == "no_renorm":
            return j == 0
        return j == nrep or (j if j < nrep else j - nrep) % renorm == 0

    for t in range(T):
        prev = gam
        gam = alpha[t] if fresh(t) else gam * alpha[t]
        inv_max = max(inv_max, float(np.max(1.0 / gam)))
        g_use = prev if (slip == "gamma_prev" and not fresh(t)) else gam
        rq = 1.0 / np.sqrt(q[t] @ q[t] + eps)
        rk = 1.0 / np.sqrt(k[t] @ k[t] + eps)
        pk = St.T @ (g_use * k[t])
        pq = St.T @ (g_use * q[t])
        e = v[t] - rk * pk
        if t >= nrep:
            o = rq * pq
            if slip != "no_output_term":
                o = o + beta[t] * (rq * rk * (q[t] @ k[t])) * e
            outs.append(o)
        kin = gam * k[t] if slip == "update_gamma" else k[t] / gam
        St = St + np.outer(kin, beta[t] * rk * e)
        if (t + 1 < T and fresh(t + 1)) or t + 1 == nrep:
            St = gam[:, None] * St  # S = Gamma S~, and Gamma restarts at the next token
        if t + 1 == nrep:
            stored = St.copy()
    return (np.array(outs).reshape(T - nrep, E), stored, inv_max)
