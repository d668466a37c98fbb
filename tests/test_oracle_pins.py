"""Pins of the fp64 oracle to facts outside itself.

Each test ties the oracle to the mathematics or to the canopy page
(projects.dotslasha.me/p/canopy.md): the sequential recurrence on a chain,
brute force on every small tree, a hand-derived T = 1 formula, the invariants
the page and the rule imply, and nilpotency of G ("The tree closed form").
"""

import itertools

import numpy as np
import pytest

import oracle
from oracle.closed_form import build_G_C
from synth import trees


def _inputs(rng, T, H, dk, dv, amin=0.01):
    q = rng.standard_normal((T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    a = rng.uniform(amin, 1.0, (T, H))
    b = rng.uniform(0.0, 1.0, (T, H))
    S0 = 0.5 * rng.standard_normal((H, dv, dk))
    return q, k, v, a, b, S0


def test_chain_equals_sequential_recurrence():
    """A chain is the plain recurrence (page: "The gated delta rule")."""
    rng = np.random.default_rng(11)
    T, H, dk, dv = 40, 3, 32, 24
    q, k, v, a, b, S0 = _inputs(rng, T, H, dk, dv)
    o, S = oracle.replay(trees.chain(T), q, k, v, a, b, S0)
    for h in range(H):
        oc, Sc = oracle.chain_recurrence(q[:, h], k[:, h], v[:, h], a[:, h], b[:, h], S0[h].T)
        assert np.abs(o[:, h] - oc).max() <= 1e-12
        assert np.abs(S[-1, h] - Sc.T).max() <= 1e-12


def _all_trees(T):
    for tail in itertools.product(*[range(i) for i in range(1, T)]):
        yield np.array((-1,) + tail, dtype=np.int32)


def test_brute_force_every_tree_up_to_8_nodes():
    """Every parent array with parent[i] < i for T = 1..8 (5,914 trees)."""
    rng = np.random.default_rng(5)
    q, k, v, a, b, S0 = _inputs(rng, 8, 1, 4, 3)
    count = 0
    for T in range(1, 9):
        for p in _all_trees(T):
            o, S = oracle.replay(p, q[:T], k[:T], v[:T], a[:T], b[:T], S0)
            ob, Sb = oracle.brute_force(p, q[:T], k[:T], v[:T], a[:T], b[:T], S0)
            assert np.abs(o - ob).max() <= 1e-12, p
            assert np.abs(S - Sb).max() <= 1e-12, p
            count += 1
    assert count == 5914


def test_closed_form_single_node():
    """T = 1: o0 = a0 S0 q0 + (k0.q0) b0 (v0 - a0 S0 k0), from the rule."""
    rng = np.random.default_rng(2)
    q, k, v, a, b, S0 = _inputs(rng, 1, 1, 16, 8)
    q0, k0, v0, a0, b0, S = q[0, 0], k[0, 0], v[0, 0], a[0, 0], b[0, 0], S0[0]
    expect = a0 * S @ q0 + (k0 @ q0) * b0 * (v0 - a0 * S @ k0)
    for solver in oracle.SOLVERS:
        O, U, l = oracle.closed_form([-1], q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], S, solver)
        assert np.abs(O[0] - expect).max() <= 1e-14
    o, _ = oracle.replay([-1], q, k, v, a, b, S0)
    assert np.abs(o[0, 0] - expect).max() <= 1e-14


def test_beta_zero_gives_decayed_S0():
    """beta = 0: o_i = gamma_i S0 q_i and S_a = gamma_a S0."""
    rng = np.random.default_rng(3)
    p = trees.uniform_random(30, rng)
    q, k, v, a, b, S0 = _inputs(rng, 30, 2, 16, 16)
    b[:] = 0
    o, S = oracle.replay(p, q, k, v, a, b, S0)
    gamma = np.exp(oracle.cumulative_log_gate(p, a))
    expect = gamma[:, :, None] * np.einsum("hvd,thd->thv", S0, q)
    assert np.abs(o - expect).max() <= 1e-13
    for leaf in trees.leaves(p):
        assert np.abs(S[leaf] - gamma[leaf][:, None, None] * S0).max() <= 1e-13
        O, U, l = oracle.closed_form(p, q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], S0[0])
        assert np.abs(U).max() == 0.0


def test_identical_sibling_subtrees_identical_outputs():
    """Two siblings with the same inputs (and identical subtrees under them)
    see the same root path values, so their outputs are bitwise equal."""
    rng = np.random.default_rng(4)
    # root 0 -> 1 -> {2, 5}; 2 -> {3, 4}; 5 -> {6, 7}; subtrees of 2 and 5 equal
    p = np.array([-1, 0, 1, 2, 2, 1, 5, 5], dtype=np.int32)
    q, k, v, a, b, S0 = _inputs(rng, 8, 2, 8, 8)
    for src, dst in ((2, 5), (3, 6), (4, 7)):
        for x in (q, k, v, a, b):
            x[dst] = x[src]
    o, S = oracle.replay(p, q, k, v, a, b, S0)
    for src, dst in ((2, 5), (3, 6), (4, 7)):
        assert (o[src] == o[dst]).all() and (S[src] == S[dst]).all()


def test_homogeneity():
    """o(cV, cS0) = c o(V, S0): the rule is linear in (V, S0) jointly."""
    rng = np.random.default_rng(6)
    p = trees.uniform_random(25, rng)
    q, k, v, a, b, S0 = _inputs(rng, 25, 2, 16, 8)
    o1, _ = oracle.replay(p, q, k, v, a, b, S0)
    o2, _ = oracle.replay(p, q, k, 3.0 * v, a, b, 3.0 * S0)
    assert np.abs(o2 - 3.0 * o1).max() <= 1e-12


@pytest.mark.parametrize("order_name", ["dfs", "level"])
def test_relabelling_invariance(order_name):
    """Any topological order gives the same per-node outputs
    (page: "Any topological order works")."""
    rng = np.random.default_rng(7)
    p = trees.uniform_random(60, rng)
    q, k, v, a, b, S0 = _inputs(rng, 60, 2, 16, 12)
    order = trees.dfs_preorder(p) if order_name == "dfs" else trees.level_order(p)
    p2 = trees.relabel(p, order)
    o1, _ = oracle.replay(p, q, k, v, a, b, S0)
    o2, _ = oracle.replay(p2, q[order], k[order], v[order], a[order], b[order], S0)
    assert np.abs(o2 - o1[order]).max() <= 1e-13
    O1, _, _ = oracle.closed_form(p, q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], S0[0])
    O2, _, _ = oracle.closed_form(p2, q[order, 0], k[order, 0], v[order, 0], a[order, 0],
                                  b[order, 0], S0[0])
    assert np.abs(O2 - O1[order]).max() <= 1e-12


@pytest.mark.parametrize("fam,T", [("chain", 17), ("top3", 40), ("random", 64), ("skewed", 64),
                                   ("top4", 341)])
def test_nilpotency(fam, T):
    """G^(d+1) = 0 exactly and G^d != 0 (page: "Nilpotency")."""
    rng = np.random.default_rng(T)
    p = trees.family(fam, T, rng)
    d = trees.tree_depth(p)
    q, k, v, a, b, S0 = _inputs(rng, T, 1, 8, 4, amin=0.5)
    G, C, l, P = build_G_C(p, q[:, 0], k[:, 0], a[:, 0], b[:, 0])
    Gd = np.linalg.matrix_power(G, d)
    assert np.abs(Gd).max() > 0
    assert (Gd @ G == 0).all()


def test_level_order_zero_diagonal_blocks():
    """In level order the block of G between nodes of equal depth is zero."""
    rng = np.random.default_rng(8)
    p = trees.uniform_random(80, rng)
    p = trees.relabel(p, trees.level_order(p))
    q, k, v, a, b, S0 = _inputs(rng, 80, 1, 8, 4)
    G, _, _, _ = build_G_C(p, q[:, 0], k[:, 0], a[:, 0], b[:, 0])
    dep = trees.node_depths(p)
    for L in range(dep.max() + 1):
        rows = np.nonzero(dep == L)[0]
        assert (G[np.ix_(rows, rows)] == 0).all()


def test_commit_every_leaf_equals_replay_state():
    """S_a from the pseudo-values equals the replayed state, for every leaf
    and for interior nodes too (page: "M1" acceptance, 1e-10)."""
    rng = np.random.default_rng(9)
    for fam, T in (("random", 100), ("top4", 85), ("skewed", 64), ("chain", 30)):
        p = trees.family(fam, T, rng)
        q, k, v, a, b, S0 = _inputs(rng, T, 2, 32, 16)
        _, S = oracle.replay(p, q, k, v, a, b, S0)
        U = np.stack([oracle.closed_form(p, q[:, h], k[:, h], v[:, h], a[:, h], b[:, h], S0[h])[1]
                      for h in range(2)], axis=1)
        for node in range(T):
            Sa = oracle.commit(p, node, k, a, U, S0)
            assert np.abs(Sa - S[node]).max() <= 1e-10


def test_grouped_value_heads_read_their_key_head():
    """HV value heads on H key heads (page: "Qwen3.5-9B shapes", grouped value
    attention): value head j is the single-head rule run with key head
    j // (HV / H); its state and output match a run of that head alone."""
    rng = np.random.default_rng(21)
    T, H, HV, dk, dv = 30, 2, 6, 16, 8
    p = trees.family("random", T, rng)
    q, k, _, _, _, _ = _inputs(rng, T, H, dk, dv)
    _, _, v, a, b, S0 = _inputs(rng, T, HV, dk, dv)
    o, S = oracle.replay(p, q, k, v, a, b, S0)
    assert o.shape == (T, HV, dv) and S.shape == (T, HV, dv, dk)
    for j in range(HV):
        h = j // (HV // H)
        oj, Sj = oracle.replay(p, q[:, [h]], k[:, [h]], v[:, [j]], a[:, [j]], b[:, [j]], S0[[j]])
        assert np.abs(o[:, j] - oj[:, 0]).max() <= 1e-13
        assert np.abs(S[:, j] - Sj[:, 0]).max() <= 1e-13
    # two value heads of one key head with the same values, gates and state agree
    v2, a2, b2, S02 = v.copy(), a.copy(), b.copy(), S0.copy()
    v2[:, 1], a2[:, 1], b2[:, 1], S02[1] = v[:, 0], a[:, 0], b[:, 0], S0[0]
    o2, _ = oracle.replay(p, q, k, v2, a2, b2, S02)
    assert np.array_equal(o2[:, 0], o2[:, 1])
    # and the commit of every node reads the same key heads
    U = np.stack([oracle.closed_form(p, q[:, j // 3], k[:, j // 3], v[:, j], a[:, j], b[:, j], S0[j])[1]
                  for j in range(HV)], axis=1)
    for node in (0, T // 2, T - 1):
        assert np.abs(oracle.commit(p, node, k, a, U, S0) - S[node]).max() <= 1e-10
    with pytest.raises(ValueError):
        oracle.replay(p, q, k, v[:, :5], a[:, :5], b[:, :5], S0[:5])


def test_q_scale_scales_the_output_only():
    """o_i = S_i (s q_i) is linear in q while the states do not depend on q
    (page: "The gated delta rule", the scale on q)."""
    rng = np.random.default_rng(22)
    T, H, dk, dv = 25, 2, 16, 8
    p = trees.family("top2", T, rng)
    q, k, v, a, b, S0 = _inputs(rng, T, H, dk, dv)
    o1, S1 = oracle.replay(p, q, k, v, a, b, S0)
    o2, S2 = oracle.replay(p, q, k, v, a, b, S0, scale=1.0 / np.sqrt(dk))
    assert np.abs(o2 - o1 / np.sqrt(dk)).max() <= 1e-13
    assert np.array_equal(S1, S2)


@pytest.mark.parametrize("fam,T", [("random", 1), ("random", 37), ("chain", 70), ("skewed", 90),
                                   ("top4", 128)])
def test_closed_form_heads_matches_replay(fam, T):
    """The head-vectorised closed form (the round trip's per-stream check)
    equals the replay, the definition, on every head, with grouped value
    heads and a q scale (canopy page, "The tree closed form"; the head layout
    of "Qwen3.5-9B shapes")."""
    rng = np.random.default_rng(T)
    p = trees.family(fam, T, rng)
    q, k, _, _, _, _ = _inputs(rng, T, 2, 16, 12)
    _, _, v, a, b, S0 = _inputs(rng, T, 4, 16, 12)
    o, _ = oracle.replay(p, q, k, v, a, b, S0, keep_states=False, scale=0.3)
    O, U, l = oracle.closed_form_heads(p, q, k, v, a, b, S0, scale=0.3)
    assert np.abs(O - o).max() <= 1e-10 * max(1.0, np.abs(o).max())
    # U and l are the per-head closed form's
    for h in range(4):
        O1, U1, l1 = oracle.closed_form(p, 0.3 * q[:, h // 2], k[:, h // 2], v[:, h], a[:, h], b[:, h], S0[h])
        assert np.abs(U[:, h] - U1).max() <= 1e-10 * max(1.0, np.abs(U1).max())
        assert np.abs(l[:, h] - l1).max() <= 1e-12


def _preorder_by_definition(parent):
    """Pre-order by recursion on the definition: a node, then each child's
    subtree in increasing child index."""
    T = len(parent)
    out = []

    def visit(n):
        out.append(n)
        for c in range(n + 1, T):
            if parent[c] == n:
                visit(c)
    visit(0)
    return out


@pytest.mark.parametrize("fam,T", [("chain", 12), ("top3", 40), ("random", 64), ("skewed", 50)])
def test_dfs_preorder(fam, T):
    """The oracle's DFS pre-order equals the recursive definition, puts every
    parent before its children and keeps every subtree contiguous."""
    p = trees.family(fam, T, np.random.default_rng(T))
    order = oracle.dfs_preorder(p)
    assert list(order) == _preorder_by_definition(p)
    pos = np.empty(T, int)
    pos[order] = np.arange(T)
    depth = oracle.depths(p)
    for i in range(1, T):
        assert pos[p[i]] < pos[i]
    for n in range(T):   # the subtree of n occupies pos[n] .. pos[n] + size - 1
        sub = [i for i in range(T) if n in oracle.root_path(p, i)]
        assert sorted(pos[sub]) == list(range(pos[n], pos[n] + len(sub)))
    assert depth[order[0]] == 0
