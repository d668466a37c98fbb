"""Commit: the accepted node's state from the pseudo-values.

canopy page, "The tree closed form" (last line of the system) and "What the
commit kernel stores", in the (dv, dk) orientation:
    S_a = P_a S0 + sum_{j in path(a)} exp(l_a - l_j) u_j k_j^T
"""

from __future__ import annotations

import numpy as np

from .replay import value_heads
from .tree import cumulative_log_gate, root_path, validate_parent


def commit(parent, a: int, k, alpha, U, S0):
    """One stream, all heads.  k [T, H, dk] (key heads); alpha [T, HV];
    U [T, HV, dv]; S0 [HV, dv, dk].  Returns S_a [HV, dv, dk]; value head j
    reads key head j // (HV / H), as in ``replay``."""
    p = validate_parent(parent)
    l = cumulative_log_gate(p, alpha)                      # [T, HV]
    U = np.asarray(U, np.float64)
    k = value_heads(k, U.shape[1])
    S = np.exp(l[a])[:, None, None] * np.asarray(S0, np.float64)
    for j in root_path(p, a):
        w = np.exp(l[a] - l[j])                            # [H]
        S = S + w[:, None, None] * U[j][:, :, None] * k[j][:, None, :]
    return S


def commit_batch(parent, accepted, k, alpha, U, S0):
    return np.stack([commit(parent[b], int(accepted[b]), k[b], alpha[b], U[b], S0[b])
                     for b in range(len(parent))])
