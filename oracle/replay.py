"""The definition: the gated delta rule run along every node's root path.

canopy page, "The gated delta rule" (TreeWY's d_v x d_k form) and "M1: Oracle
and tree generators" (the per-node replay).  For each node i in index order:
    Sp  = S0 if parent(i) = -1 else S_parent(i)
    S_i = alpha_i * Sp @ (I - beta_i k_i k_i^T) + beta_i v_i k_i^T
    o_i = S_i @ q_i
All arithmetic in float64.  Sp @ (I - beta k k^T) is evaluated as the equal
Sp - beta (Sp k) k^T, which avoids forming the dk x dk matrix.

Heads (canopy page, "Qwen3.5-9B shapes" and "Design decisions", memory
layout): q and k have H key heads, v, alpha, beta and S0 have HV value
heads, HV a multiple of H, and key head h serves value heads h * HV/H ..
(h + 1) * HV/H - 1 (grouped value attention).  q is multiplied by ``scale``
before use (the page's "The gated delta rule": the default scale on q is
1/sqrt(dk); 1 reproduces the unscaled rule).
"""

from __future__ import annotations

import numpy as np

from .tree import validate_parent


def value_heads(x, HV: int):
    """[T, H, d] per key head -> [T, HV, d] per value head: value head j reads
    key head j // (HV / H)."""
    x = np.asarray(x, np.float64)
    H = x.shape[1]
    if HV % H:
        raise ValueError(f"value heads {HV} are not a multiple of key heads {H}")
    return np.repeat(x, HV // H, axis=1)


def replay(parent, q, k, v, alpha, beta, S0, keep_states: bool = True, scale: float = 1.0):
    """One stream, all heads.

    parent [T]; q, k [T, H, dk]; v [T, HV, dv]; alpha, beta [T, HV];
    S0 [HV, dv, dk].  Returns (o [T, HV, dv], S [T, HV, dv, dk] or None).
    """
    p = validate_parent(parent)
    v = np.asarray(v, np.float64)
    HV = v.shape[1]
    q = value_heads(q, HV) * float(scale)
    k = value_heads(k, HV)
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


def replay_batch(parent, q, k, v, alpha, beta, S0, keep_states: bool = False, scale: float = 1.0):
    """B streams (one tree each); shapes as in ``replay`` with a leading B."""
    outs, states = [], []
    for bb in range(len(parent)):
        o, S = replay(parent[bb], q[bb], k[bb], v[bb], alpha[bb], beta[bb], S0[bb], keep_states, scale)
        outs.append(o)
        states.append(S)
    return np.stack(outs), (np.stack(states) if keep_states else None)
