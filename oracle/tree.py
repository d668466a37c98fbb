"""Tree bookkeeping for the oracle (its own, shared with nothing).

canopy page, "The tree closed form": nodes 0..T-1 are numbered so that every
parent precedes its child, parent(0) = -1; A(i) is the set of strict ancestors
of i and path(i) = A(i) + {i}; the depth d of the tree is the largest |A(i)|.
The cumulative log gate is l_i = log(alpha_i) + l_parent(i), with the value 0
standing for the root's parent.
"""

from __future__ import annotations

import numpy as np


def validate_parent(parent) -> np.ndarray:
    p = np.asarray(parent, dtype=np.int64)
    if p.ndim != 1 or p.size < 1:
        raise ValueError("parent must be a non-empty 1-D array")
    if p[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    for i in range(1, p.size):
        if not (0 <= p[i] < i):
            raise ValueError(f"parent[{i}] = {p[i]} is not in [0, {i})")
    return p


def root_path(parent, i: int) -> list:
    """path(i) listed from the root down to i."""
    out = []
    while i >= 0:
        out.append(int(i))
        i = int(parent[i])
    return out[::-1]


def depths(parent) -> np.ndarray:
    """|A(i)| for every node, by walking each root path."""
    return np.array([len(root_path(parent, i)) - 1 for i in range(len(parent))], dtype=np.int64)


def strict_ancestor_mask(parent) -> np.ndarray:
    """M[i, j] = True iff j is a strict ancestor of i."""
    T = len(parent)
    M = np.zeros((T, T), dtype=bool)
    for i in range(T):
        for j in root_path(parent, i)[:-1]:
            M[i, j] = True
    return M


def cumulative_log_gate(parent, alpha) -> np.ndarray:
    """l_i = sum of log(alpha_j) over j in path(i), in float64.

    alpha may carry trailing head axes: shape [T] or [T, H]."""
    a = np.asarray(alpha, dtype=np.float64)
    la = np.log(a)
    l = np.zeros_like(la)
    for i in range(len(parent)):
        l[i] = la[i] + (l[parent[i]] if parent[i] >= 0 else 0.0)
    return l


def dfs_preorder(parent) -> np.ndarray:
    """Depth-first pre-order from the root, children visited in increasing
    index order: order[pos] = the node at position pos (canopy page,
    "Design decisions", tree order: subtrees contiguous)."""
    p = validate_parent(parent)
    kids = [[] for _ in range(p.size)]
    for i in range(1, p.size):
        kids[p[i]].append(i)
    out, stack = [], [0]
    while stack:
        n = stack.pop()
        out.append(n)
        stack.extend(reversed(kids[n]))       # the smallest child is visited first
    return np.array(out, dtype=np.int64)
