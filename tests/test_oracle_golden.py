"""The oracle against the figures the canopy page prints (tests/golden/).

canopy page, "Verification of the formulas": on six named trees at d_k 16/32,
d_v 12/16, beta in (0.05, 0.95), alpha in (0.5, 0.999), five solvers matched
the per-path oracle to 8e-16 or better, the commit to 7e-16, the fp32 closed
form to 3e-7; on a 64-node chain with alpha = 0.05 naive fp32 ratios P_i/P_j
gave 630 non-finite values while the log-space form stayed within 1.4e-7.

The page gives neither seeds nor the scale of v and S0, so the fp64 and fp32
figures are checked as orders of magnitude on our own seeded draws of the
same setup (v, S0 ~ N(0, 1)), normalised by the largest reference value, with
the margin stated at each assert.  The 630 count has no free input and is
checked exactly: it is reproduced when the fp32 cumulative products are
flushed to zero below the smallest normal number (gradual underflow gives
465), and is counted over the inclusive ancestor pairs j in path(i).
"""

import json
import os

import numpy as np
import pytest

import oracle
from oracle.closed_form import naive_ratio_gamma
from synth import trees

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))
FIG = GOLD["verification_of_the_formulas"]


def _mk(rng, T, dk, dv):
    q = rng.standard_normal((T, 1, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, 1, dv))
    a = rng.uniform(*FIG["setup"]["alpha"], (T, 1))
    b = rng.uniform(*FIG["setup"]["beta"], (T, 1))
    S0 = rng.standard_normal((1, dv, dk))
    return q, k, v, a, b, S0


def _named_trees(rng):
    p40 = trees.uniform_random(40, rng)
    sp = list(range(-1, 48))                      # spine of 49 nodes: depth 48
    while len(sp) < 64:
        sp.append(int(rng.integers(0, 49)))
    sp = np.array(sp, np.int32)
    out = {
        "rand40_bfs": trees.relabel(p40, trees.level_order(p40)),
        "rand40_dfs": trees.relabel(p40, trees.dfs_preorder(p40)),
        "chain12": trees.chain(12),
        "top4_128": trees.topk(128, 4),
        "top4_256": trees.topk(256, 4),
        "skew64": trees.relabel(sp, trees.dfs_preorder(sp)),
    }
    assert trees.tree_depth(out["skew64"]) == 48
    return out


@pytest.mark.parametrize("dk,dv", [(16, 12), (32, 16)])
def test_six_named_trees(dk, dv):
    rng = np.random.default_rng(dk)
    for name, p in _named_trees(rng).items():
        T = len(p)
        q, k, v, a, b, S0 = _mk(rng, T, dk, dv)
        o, S = oracle.replay(p, q, k, v, a, b, S0)
        scale = np.abs(o).max()
        for s in oracle.SOLVERS:
            O, U, _ = oracle.closed_form(p, q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], S0[0], s)
            # a few fp64 ulps: page figure with a 4x margin for unknown inputs
            assert np.abs(O - o[:, 0]).max() / scale <= 4 * FIG["solver_max_err"], (name, s)
        for node in range(T):
            Sa = oracle.commit(p, node, k, a, U[:, None], S0)
            assert np.abs(Sa - S[node]).max() / np.abs(S[node]).max() <= 8 * FIG["commit_max_err"]
        O32, _, _ = oracle.closed_form(p, q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], S0[0],
                                       "fwdsub", np.float32)
        assert np.abs(O32 - o[:, 0]).max() / scale <= 4 * FIG["fp32_closed_form_max_err"], name


def test_naive_ratio_nonfinite_count_is_630():
    T, alpha = FIG["stability_chain_T"], FIG["stability_alpha"]
    p = trees.chain(T)
    a = np.full(T, alpha, np.float32)
    g_ftz, mask = naive_ratio_gamma(p, a, flush_subnormals=True)
    assert int((~np.isfinite(g_ftz[mask])).sum()) == FIG["naive_fp32_ratio_nonfinite_count"]
    g_ieee, _ = naive_ratio_gamma(p, a, flush_subnormals=False)
    assert int((~np.isfinite(g_ieee[mask])).sum()) == 465


@pytest.mark.parametrize("dk,dv", [(16, 12), (32, 16)])
def test_log_space_fp32_stays_finite_on_alpha_005_chain(dk, dv):
    rng = np.random.default_rng(100 + dk)
    T = FIG["stability_chain_T"]
    q, k, v, a, b, S0 = _mk(rng, T, dk, dv)
    a[:] = FIG["stability_alpha"]
    p = trees.chain(T)
    o, _ = oracle.replay(p, q, k, v, a, b, S0)
    O32, _, _ = oracle.closed_form(p, q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0], S0[0],
                                   "fwdsub", np.float32)
    assert np.isfinite(O32).all()
    # page: within 1.4e-7; 2x margin for unknown inputs
    assert np.abs(O32 - o[:, 0]).max() <= 2 * FIG["logspace_fp32_max_err"]


def test_full_top4_tree_size():
    g = GOLD["nilpotency"]["full_top4_nodes_at_depth_4"]
    assert sum(4 ** L for L in range(5)) == g
    assert trees.tree_depth(trees.topk(g, 4)) == 4
