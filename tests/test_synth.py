"""Input generators: valid trees, the stated family readings, bf16 rounding."""

import numpy as np
import pytest

import synth
from synth import trees


def _valid(p):
    assert p[0] == -1
    assert all(0 <= p[i] < i for i in range(1, len(p)))


@pytest.mark.parametrize("fam", ["chain", "top2", "top4", "top8", "skewed", "random"])
@pytest.mark.parametrize("T", [1, 3, 8, 64, 256])
def test_families_valid(fam, T):
    p = trees.family(fam, T, np.random.default_rng(T))
    assert len(p) == T
    _valid(p)


def test_family_shapes():
    assert trees.tree_depth(trees.chain(256)) == 255
    assert trees.tree_depth(trees.topk(341, 4)) == 4          # full top-4 tree of depth 4
    assert trees.tree_depth(trees.topk(342, 4)) == 5
    p = trees.skewed(64, np.random.default_rng(0))
    assert trees.tree_depth(p) >= 47                           # spine of 48 nodes
    assert (trees.dfs_preorder(p) == np.arange(64)).all()     # already DFS numbered


def test_schedule_421_tree():
    # root + 4 + 8 = 13 nodes, then 3 nodes of the third level in BFS order
    p = trees.schedule_tree(16, (4, 2, 1))
    assert list(p[:5]) == [-1, 0, 0, 0, 0]
    assert list(p[5:13]) == [1, 1, 2, 2, 3, 3, 4, 4]
    assert list(p[13:]) == [5, 6, 7]
    assert trees.tree_depth(p) == 3


def test_relabel_orders():
    rng = np.random.default_rng(3)
    p = trees.uniform_random(50, rng)
    for order in (trees.dfs_preorder(p), trees.level_order(p)):
        q = trees.relabel(p, order)
        _valid(q)
        assert sorted(trees.node_depths(q)) == sorted(trees.node_depths(p))
    d = trees.node_depths(trees.relabel(p, trees.level_order(p)))
    assert (np.diff(d) >= 0).all()


def test_random_depth_range():
    rng = np.random.default_rng(1)
    for _ in range(20):
        assert 4 <= trees.tree_depth(trees.uniform_random_depth(64, rng, 4, 20)) <= 20


def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 3
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]       # ties
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert (synth.round_bf16(x).view(np.uint32) == ref.view(np.uint32)).all()


def test_value_distributions():
    x = synth.config_inputs(2)
    assert x["q"].shape == (16, 64, 16, 128) and x["S0"].shape == (16, 16, 128, 128)
    n = np.linalg.norm(x["q"].astype(np.float64), axis=-1)
    assert np.abs(n - 1).max() < 1e-2                          # unit rows up to bf16 rounding
    assert (x["g"] > 0).all() and (x["g"] < 1).all()
    assert (x["beta"] > 0).all() and (x["beta"] < 1).all()
    assert abs(x["S0"].std() - 0.1) < 1e-3
    assert (synth.round_bf16(x["v"]) == x["v"]).all()
    for b in range(16):
        assert 4 <= trees.tree_depth(x["parent"][b]) <= 20
    y = synth.config_inputs(2)
    assert all((x[n] == y[n]).all() for n in ("q", "k", "v", "g", "beta", "S0", "parent"))
