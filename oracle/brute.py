"""Brute force: every node's root path run as a fresh chain.

canopy page, "The tree closed form": node i's output is what the recurrence
gives after the tokens of path(i), starting from the committed state S0.  Each
path is replayed from scratch with ``chain_recurrence`` (the d_k x d_v form),
nothing is shared between nodes.
"""

from __future__ import annotations

import numpy as np

from .chain import chain_recurrence
from .tree import root_path, validate_parent


def brute_force(parent, q, k, v, alpha, beta, S0):
    """One stream.  Shapes as in ``replay.replay``; S0 is [H, dv, dk].

    Returns (o [T, H, dv], S [T, H, dv, dk]) with S in the (dv, dk) layout."""
    p = validate_parent(parent)
    T, H, _ = np.shape(q)
    dv = np.shape(v)[-1]
    dk = np.shape(q)[-1]
    o = np.zeros((T, H, dv))
    S = np.zeros((T, H, dv, dk))
    for i in range(T):
        path = root_path(p, i)
        for h in range(H):
            oo, Sf = chain_recurrence(q[path, h], k[path, h], v[path, h],
                                      np.asarray(alpha)[path, h], np.asarray(beta)[path, h],
                                      np.asarray(S0[h], np.float64).T)
            o[i, h] = oo[-1]
            S[i, h] = Sf.T
    return o, S
