"""Tree-aware short causal convolution and its state commit.

canopy page, "M7: Benchmarks, the crossover, and the stretch goal" (the
end-to-end stretch run): the short causal convolution (kernel size 4) before
each GDN layer must follow each node's root path, and commit must update the
convolution state with the accepted tokens.  Written out (the plainest
reading; the page gives no formula):

  A sequence's causal depthwise convolution of kernel K is
      y_t[c] = act(bias[c] + sum_{j=0..K-1} w[c][j] * x_{t-K+1+j}[c]),
  so w[c][K-1] weighs the current token.  In a tree the tokens before node i
  are its ancestors, nearest first: a_0(i) = i, a_m(i) = parent(a_{m-1}(i)),
  and above the root come the committed sequence's last K-1 inputs, the
  convolution state (state[c][K-2] the newest, state[c][0] the oldest):
      y_i[c] = act(bias[c] + sum_{j} w[c][j] * X(i, K-1-j)[c]),
      X(i, m) = x_{a_m(i)} for m <= depth(i), else state[c][K-1-(m-depth(i))].
  Committing node a appends path(a) (root first) to the sequence: the new
  state is the last K-1 inputs of (state ++ path(a)); a = -1 keeps it.
  act is the identity or SiLU (x * sigmoid(x)).

Everything in float64 on the float64 upcast of the inputs.
"""

from __future__ import annotations

import numpy as np

from .tree import root_path, validate_parent


def _act(y, act: str):
    if act == "none":
        return y
    if act == "silu":
        return y / (1.0 + np.exp(-y))
    raise ValueError(f"unknown activation {act}")


def tree_conv(parent, x, state, w, bias=None, act: str = "none"):
    """One stream.  parent [T]; x [T, C]; state [C, K-1]; w [C, K];
    bias [C] or None.  Returns y [T, C]."""
    p = validate_parent(parent)
    x = np.asarray(x, np.float64)
    state = np.asarray(state, np.float64)
    w = np.asarray(w, np.float64)
    T, C = x.shape
    K = w.shape[1]
    b = np.zeros(C) if bias is None else np.asarray(bias, np.float64)
    y = np.empty((T, C))
    for i in range(T):
        path = root_path(p, i)                       # root first, i last
        seq = np.concatenate([state.T, x[path]], 0)  # [K-1 + depth + 1, C], oldest first
        window = seq[-K:]                            # the K most recent inputs, oldest first
        y[i] = _act(b + (w.T * window).sum(0), act)
    return y


def conv_commit(parent, a: int, x, state):
    """One stream: the state after accepting node a.  x [T, C];
    state [C, K-1].  Returns [C, K-1]."""
    state = np.asarray(state, np.float64)
    if a < 0:
        return state.copy()
    p = validate_parent(parent)
    x = np.asarray(x, np.float64)
    seq = np.concatenate([state.T, x[root_path(p, a)]], 0)
    return seq[-state.shape[1]:].T.copy()


def tree_conv_batch(parent, x, state, w, bias=None, act: str = "none"):
    return np.stack([tree_conv(parent[b], x[b], state[b], w, bias, act) for b in range(len(parent))])


def conv_commit_batch(parent, accepted, x, state):
    return np.stack([conv_commit(parent[b], int(accepted[b]), x[b], state[b]) for b in range(len(parent))])
