"""GPU parity of the solve variants (canopy page, "The tree closed form":
nilpotency and the squaring form; "Design decisions": the Neumann series and
the split design) against the fp64 oracle replay, through the C ABI.

Every variant must give the same o (and, through the commit, the same
accepted state) as the default blocked substitution, within the bf16-input
tolerance (max |x - x_ref| / rms(x_ref) <= 1e-2).
"""

import numpy as np
import pytest
import torch

import synth
from synth import trees
from tests.gpu_helpers import TOL_BF16, oracle_outputs, rel_err, run_verify, to_device

pytestmark = pytest.mark.gpu

VARIANTS = ["neumann", "squaring", "split"]


def _inputs(T, fam, B=2, H=4, seed=0):
    rng = np.random.default_rng(seed + 6007 * T)
    parents = [trees.family(fam, T, rng) for _ in range(B)]
    return synth.make_inputs(parents, H, 128, 128, True, case=94, rnd=seed)


def _check(lib, inp, solve, o_dtype=torch.float32, scale=1.0, accept=None):
    o_ref, S_ref = oracle_outputs(inp, keep_states=True, scale=scale)
    dev = to_device(inp, bf16=True)
    o, ws, err = run_verify(lib, dev, solve=solve, o_dtype=o_dtype, scale=scale)
    assert err == 0
    on = o.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(on).all()
    if o_dtype == torch.bfloat16:
        # the bound plus the rounding of o to bf16 (half an ulp, 2^-8 relative)
        excess = np.maximum(np.abs(on - o_ref) - 2.0 ** -8 * np.abs(o_ref), 0.0)
        eo = float(excess.max() / np.sqrt((o_ref ** 2).mean()))
    else:
        eo = rel_err(on, o_ref)
    assert eo <= TOL_BF16, eo
    B, T = inp["parent"].shape
    a = np.full(B, T - 1, np.int32) if accept is None else np.asarray(accept, np.int32)
    Sn = lib.commit(torch.from_numpy(a).cuda(), dev["S0"], dev["k"], dev["parent"], ws)
    assert lib.read_device_error(ws) == 0
    es = rel_err(Sn.cpu().numpy(), S_ref[np.arange(B), a])
    assert es <= TOL_BF16, es
    return eo, es


@pytest.mark.parametrize("solve", VARIANTS)
@pytest.mark.parametrize("fam", ["chain", "top4", "skewed", "random"])
@pytest.mark.parametrize("T", [1, 2, 17, 64, 65, 100, 129, 256])
def test_variant_matches_oracle(lib, solve, fam, T):
    _check(lib, _inputs(T, fam), solve)


@pytest.mark.parametrize("solve", VARIANTS)
def test_variant_bf16_output_and_leaf_commit(lib, solve):
    """bf16 o, and a commit to a leaf of each stream (not the last node)."""
    inp = _inputs(200, "top2", B=3)
    leaves = [int(trees.leaves(p)[0]) for p in inp["parent"]]
    _check(lib, inp, solve, o_dtype=torch.bfloat16, accept=leaves)


@pytest.mark.parametrize("solve", VARIANTS)
@pytest.mark.parametrize("T", [48, 150])
def test_variant_grouped_value_heads_and_scale(lib, solve, T):
    """Two value heads per key head, q scaled by 1/sqrt(dk)."""
    rng = np.random.default_rng(5 + T)
    parents = [trees.family("random", T, rng) for _ in range(2)]
    ik = synth.make_inputs(parents, 2, 128, 128, True, case=95)
    iv = synth.make_inputs(parents, 4, 128, 128, True, case=96)
    _check(lib, dict(iv, q=ik["q"], k=ik["k"]), solve, scale=128 ** -0.5)


@pytest.mark.parametrize("solve", VARIANTS)
def test_variant_small_gates(lib, solve):
    """A 256-node chain with every gate 0.05 (the page's stability case at
    full depth) and a random tree with gates down to 0.01."""
    inp = _inputs(256, "chain", B=1)
    inp["g"] = np.full_like(inp["g"], 0.05)
    _check(lib, inp, solve)
    inp = _inputs(256, "random", B=2, seed=1)
    inp["g"] = np.random.default_rng(3).uniform(0.01, 1.0, inp["g"].shape).astype(np.float32)
    _check(lib, inp, solve)


@pytest.mark.parametrize("solve", ["fwdsub"] + VARIANTS)
def test_level_and_dfs_order_agree(lib, solve):
    """One tree under DFS pre-order and under level order (both topological;
    canopy page, "Design decisions", tree order and tiling): each matches the
    oracle, and the outputs agree node for node after relabelling."""
    rng = np.random.default_rng(11)
    base = trees.family("random", 180, rng)
    outs = []
    for order in (trees.dfs_preorder(base), trees.level_order(base)):
        p = trees.relabel(base, order)
        inp = synth.make_inputs([p], 4, 128, 128, True, case=97)
        # the same per-node values under both labellings: node n is old node order[n]
        ref = synth.make_inputs([base], 4, 128, 128, True, case=97)
        for n in ("q", "k", "v", "g", "beta"):
            inp[n] = ref[n][:, order]
        inp["S0"] = ref["S0"]
        _check(lib, inp, solve)
        o, _, _ = run_verify(lib, to_device(inp, True), solve=solve)
        back = np.empty_like(o.cpu().numpy())
        back[:, order] = o.cpu().numpy()
        outs.append(back)
    assert rel_err(outs[0], outs[1]) <= TOL_BF16


@pytest.mark.parametrize("solve", VARIANTS)
def test_variants_want_bf16_and_d128(lib, solve):
    inp = _inputs(32, "random")
    with pytest.raises(lib.CanopyError):
        run_verify(lib, to_device(inp, bf16=False), solve=solve)
    small = synth.make_inputs([trees.family("random", 16, np.random.default_rng(0))], 2, 32, 32, True)
    with pytest.raises(lib.CanopyError):
        run_verify(lib, to_device(small, bf16=True), solve=solve)
