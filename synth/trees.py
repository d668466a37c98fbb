"""Draft-tree generators (parent arrays).

A tree of T nodes is an int32 array ``parent`` with ``parent[0] == -1`` and
``0 <= parent[i] < i`` for i >= 1: nodes are numbered in a topological order,
node 0 is the root (canopy page, "The tree closed form").  The families are the
ones the page sweeps ("Design decisions", "Where parallel stops winning", and
"M1"): chains, balanced top-k trees, skewed trees (one long spine with short
side branches), uniform random trees, and the named shapes of the papers it
summarises.

Readings where the page is silent (stated once here, used everywhere):
  * balanced top-k at size T: the complete k-ary tree numbered breadth-first
    and cut after T nodes, so parent[i] = (i - 1) // k;
  * a branching schedule (b1, b2, ...): level 1 is the root, each node of level
    L has b_L children, numbering is breadth-first, and the tree is cut after T
    nodes (the (4, 2, 1) schedule cut at 16 nodes is the batch-1 Qwen3.5-like
    layer case);
  * skewed: a spine of ceil(0.75 T) nodes, the rest as side chains of length 1
    or 2 hung from uniformly drawn spine nodes, then renumbered in DFS
    pre-order;
  * uniform random: parent[i] uniform over 0..i-1 (a random recursive tree).
"""

from __future__ import annotations

import math

import numpy as np


def _check(parent: np.ndarray) -> np.ndarray:
    parent = np.asarray(parent, dtype=np.int32)
    assert parent.ndim == 1 and parent.size >= 1
    assert parent[0] == -1
    for i in range(1, parent.size):
        assert 0 <= parent[i] < i, (i, parent[i])
    return parent


def chain(T: int) -> np.ndarray:
    """A chain of T nodes: node i's parent is i - 1 (depth T - 1)."""
    return np.arange(-1, T - 1, dtype=np.int32)


def topk(T: int, k: int) -> np.ndarray:
    """Complete k-ary tree in breadth-first numbering, cut after T nodes."""
    p = np.empty(T, dtype=np.int32)
    p[0] = -1
    for i in range(1, T):
        p[i] = (i - 1) // k
    return p


def schedule_tree(T: int, schedule) -> np.ndarray:
    """Breadth-first tree where every node of level L (root = level 1) has
    schedule[L-1] children; the last entry repeats for deeper levels.  Cut
    after T nodes."""
    p = [-1]
    frontier = [0]
    level = 0
    while len(p) < T and frontier:
        b = schedule[min(level, len(schedule) - 1)]
        nxt = []
        for node in frontier:
            for _ in range(b):
                if len(p) >= T:
                    break
                p.append(node)
                nxt.append(len(p) - 1)
        frontier = nxt
        level += 1
    assert len(p) == T, "schedule cannot reach T nodes"
    return np.asarray(p, dtype=np.int32)


def uniform_random(T: int, rng: np.random.Generator) -> np.ndarray:
    """Random recursive tree: parent[i] uniform over 0..i-1."""
    p = np.empty(T, dtype=np.int32)
    p[0] = -1
    for i in range(1, T):
        p[i] = rng.integers(0, i)
    return p


def uniform_random_depth(T: int, rng: np.random.Generator, lo: int, hi: int,
                         max_draws: int = 10000) -> np.ndarray:
    """Uniform random tree redrawn until its depth lies in [lo, hi]."""
    for _ in range(max_draws):
        p = uniform_random(T, rng)
        if lo <= tree_depth(p) <= hi:
            return p
    raise RuntimeError(f"no tree of {T} nodes with depth in [{lo}, {hi}]")


def skewed(T: int, rng: np.random.Generator) -> np.ndarray:
    """One long spine with short side chains, renumbered in DFS pre-order."""
    spine = max(1, math.ceil(0.75 * T))
    p = list(range(-1, spine - 1))
    while len(p) < T:
        host = int(rng.integers(0, spine))
        length = int(min(rng.integers(1, 3), T - len(p)))
        prev = host
        for _ in range(length):
            p.append(prev)
            prev = len(p) - 1
    p = np.asarray(p, dtype=np.int32)
    return relabel(p, dfs_preorder(p))


def node_depths(parent) -> np.ndarray:
    parent = np.asarray(parent)
    d = np.zeros(parent.size, dtype=np.int32)
    for i in range(1, parent.size):
        d[i] = d[parent[i]] + 1
    return d


def tree_depth(parent) -> int:
    """Largest number of strict ancestors of any node (0 for a single node)."""
    return int(node_depths(parent).max())


def leaves(parent) -> np.ndarray:
    parent = np.asarray(parent)
    has_child = np.zeros(parent.size, dtype=bool)
    has_child[parent[1:]] = True
    return np.nonzero(~has_child)[0].astype(np.int32)


def _children(parent):
    ch = [[] for _ in range(len(parent))]
    for i in range(1, len(parent)):
        ch[parent[i]].append(i)
    return ch


def dfs_preorder(parent) -> np.ndarray:
    """order[new_position] = old node, children visited in index order."""
    ch = _children(parent)
    order, stack = [], [0]
    while stack:
        n = stack.pop()
        order.append(n)
        stack.extend(reversed(ch[n]))
    return np.asarray(order, dtype=np.int32)


def level_order(parent) -> np.ndarray:
    """order[new_position] = old node, sorted by depth then by index."""
    d = node_depths(parent)
    return np.lexsort((np.arange(len(parent)), d)).astype(np.int32)


def relabel(parent, order) -> np.ndarray:
    """Renumber so that new node n is old node order[n]; order must be
    topological (every parent placed before its children)."""
    parent = np.asarray(parent)
    order = np.asarray(order)
    pos = np.empty_like(order)
    pos[order] = np.arange(order.size)
    newp = np.empty(order.size, dtype=np.int32)
    for n, old in enumerate(order):
        newp[n] = -1 if parent[old] < 0 else pos[parent[old]]
    return _check(newp)


def family(name: str, T: int, rng: np.random.Generator) -> np.ndarray:
    """Tree by family name: 'chain', 'top2'..'top8', 'skewed', 'random'."""
    if name == "chain":
        return chain(T)
    if name.startswith("top"):
        return topk(T, int(name[3:]))
    if name == "skewed":
        return skewed(T, rng)
    if name == "random":
        return uniform_random(T, rng)
    raise ValueError(name)
