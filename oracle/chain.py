"""Sequential gated delta rule for a chain, flash-linear-attention orientation.

canopy page, "The gated delta rule": the state has shape d_k x d_v and for
token t
    S~_t = alpha_t S_{t-1}
    u_t  = beta_t (v_t - S~_t^T k_t)
    S_t  = S~_t + k_t u_t^T
    o_t  = S_t^T q_t
Written independently of ``replay`` (other orientation, other update order) so
that a transposed operand in either one shows up as a mismatch.
"""

from __future__ import annotations

import numpy as np


def chain_recurrence(q, k, v, alpha, beta, S0_kv):
    """One head.  q, k [T, dk]; v [T, dv]; alpha, beta [T]; S0_kv [dk, dv].

    Returns (o [T, dv], final state [dk, dv])."""
    S = np.array(S0_kv, dtype=np.float64)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T = q.shape[0]
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        St = float(alpha[t]) * S
        u = float(beta[t]) * (v[t] - St.T @ k[t])
        S = St + np.outer(k[t], u)
        o[t] = S.T @ q[t]
    return o, S
