"""GPU parity of the standalone tree preparation (canopy_tree_prep) against
the oracle's tree functions.

canopy page, "The tree closed form" (A(i), path(i), depth, l_i = log alpha_i
+ l_parent(i)) and "Design decisions" (the ancestor bitmask; DFS pre-order
keeps subtrees contiguous).  Integer outputs (depth, mask, order) must match
bit for bit; l is computed from fp32 logarithms, so it is held to fp32
rounding of each term (1e-6 per term of the path, relative to |l|).
A malformed parent array is reported in the error word and read as the
sanitised tree (a parent outside [0, i) becomes 0; a root with a parent
becomes a root), and the outputs are the oracle's for that tree.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import trees

pytestmark = pytest.mark.gpu


def _pack_mask(M):
    """Boolean [T, T] strict-ancestor matrix -> uint32 words [T, ceil(T/32)]."""
    T = M.shape[0]
    W = (T + 31) // 32
    out = np.zeros((T, W), np.uint64)
    for j in range(T):
        out[:, j // 32] |= M[:, j].astype(np.uint64) << np.uint64(j % 32)
    return out.astype(np.uint32)


def _run(lib, parents, g):
    B, T = parents.shape
    HV = g.shape[-1]
    ws = lib.workspace(B, T, HV, 128)
    par = torch.from_numpy(parents.astype(np.int32)).cuda()
    gd = torch.from_numpy(g.astype(np.float32)).cuda()
    lib.tree_prep(par, gd, ws)
    err = lib.read_device_error(ws)
    v = lib.workspace_views(ws, B, T, HV, 128)
    return err, {n: x.cpu().numpy() for n, x in v.items() if n != "u"}


def _check(out, parents, g):
    B, T = parents.shape
    for b in range(B):
        p = parents[b]
        assert np.array_equal(out["depth"][b], oracle.depths(p))
        assert np.array_equal(out["mask"][b].view(np.uint32), _pack_mask(oracle.strict_ancestor_mask(p)))
        assert np.array_equal(out["order"][b], oracle.dfs_preorder(p))
        l_ref = oracle.cumulative_log_gate(p, g[b])
        tol = 1e-6 * (oracle.depths(p)[:, None] + 1) * np.maximum(1.0, np.abs(l_ref))
        assert np.all(np.abs(out["l"][b] - l_ref) <= tol)


@pytest.mark.parametrize("T", [1, 2, 31, 32, 33, 64, 65, 100, 128, 200, 255, 256])
def test_tree_prep_matches_oracle(lib, T):
    rng = np.random.default_rng(100 + T)
    fams = ["chain", "top2", "top5", "skewed", "random"]
    parents = np.stack([trees.family(f, T, rng) for f in fams])
    g = np.exp(-np.logaddexp(0, rng.standard_normal((len(fams), T, 6)))).astype(np.float32)
    err, out = _run(lib, parents, g)
    assert err == 0
    _check(out, parents, g)


def test_tree_prep_small_gates_deep_chain(lib):
    """A 256-node chain with every gate 0.01: l reaches about -1,179, and the
    fp64 sums of fp32 logarithms keep it within rounding of each term."""
    T = 256
    parents = trees.chain(T)[None]
    g = np.full((1, T, 3), 0.01, np.float32)
    err, out = _run(lib, parents, g)
    assert err == 0
    _check(out, parents, g)


def test_tree_prep_sanitises_bad_parents(lib):
    T = 100
    rng = np.random.default_rng(5)
    good = np.stack([trees.uniform_random(T, rng) for _ in range(3)])
    bad = good.copy()
    bad[0, 0] = 4             # root with a parent
    bad[1, 50] = 50           # parent[i] = i
    bad[2, 99] = 1000         # out of range
    bad[2, 7] = -3
    fixed = good.copy()
    fixed[0, 0] = -1
    fixed[1, 50] = 0
    fixed[2, 99] = 0
    fixed[2, 7] = 0
    g = np.exp(-np.logaddexp(0, rng.standard_normal((3, T, 2)))).astype(np.float32)
    err, out = _run(lib, bad, g)
    assert err & 0x1
    _check(out, fixed, g)


def test_tree_prep_bad_gate_flagged(lib):
    T = 40
    parents = trees.topk(T, 3)[None]
    g = np.full((1, T, 2), 0.5, np.float32)
    g[0, 10, 1] = 0.0
    err, _ = _run(lib, parents, g)
    assert err & 0x2
