"""Pins of the oracle's tree-aware short convolution (canopy page, "M7:
Benchmarks, the crossover, and the stretch goal": the short causal
convolution follows each node's root path; commit updates its state)."""

import numpy as np
import pytest

import oracle
from synth import trees


def _case(rng, T, C, K):
    x = rng.standard_normal((T, C))
    state = rng.standard_normal((C, K - 1))
    w = rng.standard_normal((C, K))
    bias = rng.standard_normal(C)
    return x, state, w, bias


@pytest.mark.parametrize("K", [2, 4, 6])
def test_chain_is_the_sequence_convolution(K):
    """On a chain the tree convolution is the ordinary causal depthwise
    convolution of (state ++ x), computed here by numpy's convolve."""
    rng = np.random.default_rng(K)
    T, C = 20, 5
    x, state, w, bias = _case(rng, T, C, K)
    y = oracle.tree_conv(trees.chain(T), x, state, w, bias)
    seq = np.concatenate([state.T, x], 0)
    for c in range(C):
        full = np.convolve(seq[:, c], w[c, ::-1], mode="valid")   # y_t = sum_j w[j] x_{t-K+1+j}
        assert np.abs(y[:, c] - (full + bias[c])).max() <= 1e-12


def test_tree_nodes_see_their_root_path_only():
    """Every node's output equals the chain convolution over its own root
    path; siblings with the same input agree; SiLU applies on top."""
    rng = np.random.default_rng(3)
    T, C, K = 40, 4, 4
    p = trees.family("random", T, rng)
    x, state, w, bias = _case(rng, T, C, K)
    y = oracle.tree_conv(p, x, state, w, bias, act="silu")
    for i in range(T):
        path = oracle.root_path(p, i)
        yc = oracle.tree_conv(trees.chain(len(path)), x[path], state, w, bias, act="none")[-1]
        assert np.abs(y[i] - yc / (1 + np.exp(-yc))).max() <= 1e-12
    # a sibling pair with the same input gives the same output
    kids = [i for i in range(1, T) if p[i] == 0]
    if len(kids) >= 2:
        x2 = x.copy()
        x2[kids[1]] = x2[kids[0]]
        y2 = oracle.tree_conv(p, x2, state, w, bias)
        assert np.array_equal(y2[kids[0]], y2[kids[1]])


def test_commit_appends_the_accepted_path():
    rng = np.random.default_rng(4)
    T, C, K = 30, 3, 4
    p = trees.family("top2", T, rng)
    x, state, _, _ = _case(rng, T, C, K)
    for a in (-1, 0, 1, 5, T - 1):
        new = oracle.conv_commit(p, a, x, state)
        seq = np.concatenate([state.T] + ([x[oracle.root_path(p, a)]] if a >= 0 else []), 0)
        assert np.array_equal(new, seq[-(K - 1):].T)
    # on a chain, committing node a and convolving the rest of the chain from
    # the new state gives the outputs the whole chain gave after a
    ch = trees.chain(T)
    a = 6
    w, bias = _case(np.random.default_rng(9), T, C, K)[2:]
    y1 = oracle.tree_conv(ch, x, state, w, bias)
    s2 = oracle.conv_commit(ch, a, x, state)
    y2 = oracle.tree_conv(trees.chain(T - a - 1), x[a + 1:], s2, w, bias)
    assert np.abs(y1[a + 1:] - y2).max() <= 1e-12
