"""The definition: the gated delta rule run along every node's root path.

canopy page, "The gated delta rule" (TreeWY's d_v x d_k form) and "M1: Oracle
and tree generators" (the per-node replay).  For each node i in index order:
    Sp  = S0 if parent(i) = -1 else S_parent(i)
    S_i = alpha_i * Sp @ (I - beta_i k_i k_i^T) + beta_i v_i k_i^T
    o_i = S_i @ q_i
All arithmetic in float64.  Sp @ (I - beta k k^T) is evaluated as the equal
Sp - beta (Sp k) k^T, which avoids forming the dk x dk matrix.
"""

from __future__ import annotations

import numpy as np

from .tree import validate_parent


def replay(parent, q, k, v, alpha, beta, S0, keep_states: bool = True):
    """One stream, all heads.

    parent [T]; q, k [T, H, dk]; v [T, H, dv]; alpha, beta [T, H];
    S0 [H, dv, dk].  Returns (o [T, H, dv], S [T, H, dv, dk] or None).
    """
    p = validate_parent(parent)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    a = np.asarray(alpha, np.float64)
    b = np.asarray(beta, np.float64)
    S0 = np.asarray(S0, np.float64)
    T, H, dk = q.shape
    dv = v.shape[-1]
    last_child = np.full(T, -1)
    for i in range(1, T):
        last_child[p[i]] = i
    states = {}
    S_all = np.empty((T, H, dv, dk)) if keep_states else None
    o = np.empty((T, H, dv))
    for i in range(T):
        Sp = S0 if p[i] < 0 else states[p[i]]
        Spk = np.einsum("hvd,hd->hv", Sp, k[i])                  # Sp k_i
        ai = a[i][:, None, None]
        bi = b[i][:, None, None]
        Si = ai * (Sp - bi * Spk[:, :, None] * k[i][:, None, :]) \
            + bi * v[i][:, :, None] * k[i][:, None, :]
        o[i] = np.einsum("hvd,hd->hv", Si, q[i])                 # S_i q_i
        if last_child[i] >= 0:
            states[i] = Si                       # kept until its last child is done
        if p[i] >= 0 and last_child[p[i]] == i:
            del states[p[i]]
        if keep_states:
            S_all[i] = Si
    return o, S_all


def replay_batch(parent, q, k, v, alpha, beta, S0, keep_states: bool = False):
    """B streams (one tree each); shapes as in ``replay`` with a leading B."""
    outs, states = [], []
    for bb in range(len(parent)):
        o, S = replay(parent[bb], q[bb], k[bb], v[bb], alpha[bb], beta[bb], S0[bb], keep_states)
        outs.append(o)
        states.append(S)
    return np.stack(outs), (np.stack(states) if keep_states else None)
