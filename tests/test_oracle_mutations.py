"""Planted mistakes in the oracle must turn a pin red.

Each mutation is a plausible slip (a causal triangle for the ancestor mask, a
dropped beta, a dropped own gate, a transposed state, a flipped sign, the
naive ratio, a solver one round or one factor short, a transposed inverse).  The mutated function is built here, on the CPU, from the
oracle's own pieces; the check is the one the pins use.
"""

import numpy as np

import oracle
from oracle.closed_form import SOLVERS, naive_ratio_gamma
from oracle.tree import cumulative_log_gate, strict_ancestor_mask
from synth import trees


def _inputs(seed, T, dk=16, dv=12):
    rng = np.random.default_rng(seed)
    p = trees.uniform_random(T, rng)
    q = rng.standard_normal((T, 1, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, 1, dv))
    a = rng.uniform(0.3, 1.0, (T, 1))
    b = rng.uniform(0.1, 1.0, (T, 1))
    S0 = rng.standard_normal((1, dv, dk))
    return p, q, k, v, a, b, S0


def _closed_form_variant(p, q, k, v, a, b, S0, causal=False, drop_beta=False,
                         drop_own_gate=False):
    T = len(p)
    Ms = np.tril(np.ones((T, T), bool), -1) if causal else strict_ancestor_mask(p)
    Mp = Ms | np.eye(T, dtype=bool)
    l = cumulative_log_gate(p, a)
    if drop_own_gate:
        l = l - np.log(a)
    diff = np.where(Mp, l[:, None] - l[None, :], 0.0)
    Gam = np.where(Mp, np.exp(diff), 0.0)
    bb = np.ones_like(b) if drop_beta else b
    G = np.where(Ms, bb[:, None] * Gam * (k @ k.T), 0.0)
    C = np.where(Mp, Gam * (q @ k.T), 0.0)
    P = np.exp(l)
    R = b[:, None] * (v - P[:, None] * (k @ S0.T))
    U = SOLVERS["fwdsub"](G, R, p)
    return P[:, None] * (q @ S0.T) + C @ U


def _err_vs_replay(mut):
    p, q, k, v, a, b, S0 = _inputs(1, 40)
    o, _ = oracle.replay(p, q, k, v, a, b, S0)
    O = _closed_form_variant(p, q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], S0[0], **mut)
    return np.abs(O - o[:, 0]).max()


def test_unmutated_passes():
    assert _err_vs_replay({}) <= 1e-12


def test_causal_triangle_fails():
    assert _err_vs_replay({"causal": True}) > 1e-3


def test_dropped_beta_fails():
    assert _err_vs_replay({"drop_beta": True}) > 1e-3


def test_dropped_own_gate_fails():
    assert _err_vs_replay({"drop_own_gate": True}) > 1e-3


def test_transposed_state_fails_chain_pin():
    p, q, k, v, a, b, S0 = _inputs(2, 20, dk=8, dv=8)
    o, _ = oracle.replay(trees.chain(20), q, k, v, a, b, np.swapaxes(S0, 1, 2))
    oc, _ = oracle.chain_recurrence(q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], S0[0].T)
    assert np.abs(o[:, 0] - oc).max() > 1e-3


def test_flipped_sign_fails_brute_force_pin():
    p, q, k, v, a, b, S0 = _inputs(3, 8, dk=4, dv=3)
    ob, _ = oracle.brute_force(p, q, k, v, a, b, S0)
    # replay with (I + beta k k^T) in place of (I - beta k k^T)
    S = {}
    o = np.zeros_like(ob)
    for i in range(8):
        Sp = S0[0] if p[i] < 0 else S[p[i]]
        Si = a[i, 0] * (Sp + b[i, 0] * np.outer(Sp @ k[i, 0], k[i, 0])) + b[i, 0] * np.outer(v[i, 0], k[i, 0])
        S[i] = Si
        o[i, 0] = Si @ q[i, 0]
    assert np.abs(o - ob).max() > 1e-3


def test_naive_ratio_is_not_finite():
    g, mask = naive_ratio_gamma(trees.chain(64), np.full(64, 0.05, np.float32), True)
    assert not np.isfinite(g[mask]).all()


def _solver_err(solve):
    """max |U - U_dense| of a (mutated) solver on a 40-node tree whose nodes
    share one key (k_i.k_j = 1), so that every term of the series is large
    enough to see (the identical-keys pin's inputs)."""
    rng = np.random.default_rng(4)
    p = trees.uniform_random(40, rng)
    T, dk = 40, 8
    k1 = rng.standard_normal(dk)
    k = np.tile(k1 / np.linalg.norm(k1), (T, 1))
    q = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, 6))
    a = rng.uniform(0.8, 1.0, T)
    b = rng.uniform(0.4, 0.6, T)
    S0 = 0.1 * rng.standard_normal((6, dk))
    G, C, l, P = oracle.build_G_C(p, q, k, a, b)
    R = b[:, None] * (v - P[:, None] * (k @ S0.T))
    assert int(trees.node_depths(p).max()) >= 4
    return np.abs(solve(G, R, p) - SOLVERS["dense"](G, R, p)).max()


def test_every_solver_unmutated_passes():
    for name, fn in SOLVERS.items():
        assert _solver_err(fn) <= 1e-12, name


def test_neumann_one_round_short_fails():
    def short(G, R, p):
        d = int(trees.node_depths(p).max())
        Z, U = R.copy(), R.copy()
        for _ in range(d - 1):
            Z = -(G @ Z)
            U = U + Z
        return U
    assert _solver_err(short) > 1e-6


def test_squaring_one_factor_short_fails():
    def short(G, R, p):
        d = int(trees.node_depths(p).max())
        nfac = int(np.ceil(np.log2(d + 1))) - 1
        U, Gp = R - G @ R, G
        for _ in range(1, nfac):
            Gp = Gp @ Gp
            U = U + Gp @ U
        return U
    assert _solver_err(short) > 1e-6


def test_squaring_with_a_plus_first_factor_fails():
    def plus(G, R, p):
        d = int(trees.node_depths(p).max())
        nfac = int(np.ceil(np.log2(d + 1)))
        U, Gp = R + G @ R, G
        for _ in range(1, nfac):
            Gp = Gp @ Gp
            U = U + Gp @ U
        return U
    assert _solver_err(plus) > 1e-3


def test_split_with_transposed_inverse_fails():
    def transposed(G, R, p):
        T = G.shape[0]
        W = np.zeros_like(G)
        for i in range(T):
            W[i] = -(G[i, :i] @ W[:i])
            W[i, i] += 1.0
        return W.T @ R
    assert _solver_err(transposed) > 1e-3
