"""GPU parity of the tree-aware short convolution and its state commit
(canopy page, "M7: Benchmarks, the crossover, and the stretch goal")
against the fp64 oracle on the same seeded inputs.

Tolerances: fp32 inputs, fp32 arithmetic over K taps: 1e-5 max/rms; bf16
inputs and output: the rounding of y to bf16 (half an ulp, 2^-8 of the
value) plus 1e-5."""

import numpy as np
import pytest
import torch

import oracle
from synth import trees
from tests.gpu_helpers import rel_err

pytestmark = pytest.mark.gpu


def _case(T, fam, B, C, K, bf16, seed=0):
    rng = np.random.default_rng(seed + 17 * T + K)
    parents = np.stack([trees.family(fam, T, rng) for _ in range(B)]).astype(np.int32)
    x = rng.standard_normal((B, T, C)).astype(np.float32)
    if bf16:
        x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    state = rng.standard_normal((B, C, K - 1)).astype(np.float32)
    w = (0.5 * rng.standard_normal((C, K))).astype(np.float32)
    bias = (0.1 * rng.standard_normal(C)).astype(np.float32)
    return parents, x, state, w, bias


def _dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype).contiguous()


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("T,fam,K", [(1, "chain", 4), (5, "chain", 4), (16, "top4", 4), (64, "random", 4),
                                     (64, "skewed", 2), (100, "random", 6), (256, "top2", 8)])
@pytest.mark.parametrize("act", ["none", "silu"])
def test_tree_conv_matches_oracle(lib, T, fam, K, bf16, act):
    B, C = 3, 96
    parents, x, state, w, bias = _case(T, fam, B, C, K, bf16)
    ref = oracle.tree_conv_batch(parents, x, state, w, bias, act)
    xd = _dev(x, torch.bfloat16 if bf16 else torch.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = lib.tree_conv(xd, _dev(state), _dev(w), _dev(parents, torch.int32), bias=_dev(bias), act=act, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    yn = y.float().cpu().numpy().astype(np.float64)
    if bf16:
        excess = np.maximum(np.abs(yn - ref) - 2.0 ** -8 * np.abs(ref), 0.0)
        assert excess.max() / np.sqrt((ref ** 2).mean()) <= 1e-5
    else:
        assert rel_err(yn, ref) <= 1e-5


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("T,fam,K", [(5, "chain", 4), (64, "random", 3), (200, "skewed", 8)])
def test_tree_conv_channels_not_a_multiple_of_8(lib, T, fam, K, bf16):
    """C = 100 (a multiple of 4, not of 8) takes the four-channel kernel;
    C = 104 the eight-channel one with a partial last block."""
    for C in (100, 104):
        parents, x, state, w, bias = _case(T, fam, 2, C, K, bf16, seed=C)
        ref = oracle.tree_conv_batch(parents, x, state, w, bias, "silu")
        xd = _dev(x, torch.bfloat16 if bf16 else torch.float32)
        y = lib.tree_conv(xd, _dev(state), _dev(w), _dev(parents, torch.int32), bias=_dev(bias), act="silu")
        yn = y.float().cpu().numpy().astype(np.float64)
        if bf16:
            excess = np.maximum(np.abs(yn - ref) - 2.0 ** -8 * np.abs(ref), 0.0)
            assert excess.max() / np.sqrt((ref ** 2).mean()) <= 1e-5
        else:
            assert rel_err(yn, ref) <= 1e-5


def test_tree_conv_model_width_without_bias(lib):
    """The convolution width of the pages' layer shape: q, k (16 heads) and v
    (32 heads) of 128 channels each, C = 8,192, no bias, SiLU."""
    B, T, C, K = 2, 16, 8192, 4
    parents, x, state, w, _ = _case(T, "top4", B, C, K, True, seed=5)
    ref = oracle.tree_conv_batch(parents, x, state, w, None, "silu")
    y = lib.tree_conv(_dev(x, torch.bfloat16), _dev(state), _dev(w), _dev(parents, torch.int32), act="silu")
    yn = y.float().cpu().numpy().astype(np.float64)
    excess = np.maximum(np.abs(yn - ref) - 2.0 ** -8 * np.abs(ref), 0.0)
    assert excess.max() / np.sqrt((ref ** 2).mean()) <= 1e-5


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("K", [2, 4, 8])
def test_conv_commit_matches_oracle_and_in_place(lib, K, bf16):
    B, T, C = 4, 40, 64
    parents, x, state, _, _ = _case(T, "random", B, C, K, bf16, seed=2)
    accepted = np.array([-1, 0, T - 1, int(trees.leaves(parents[3])[0])], dtype=np.int32)
    ref = oracle.conv_commit_batch(parents, accepted, x, state)
    xd = _dev(x, torch.bfloat16 if bf16 else torch.float32)
    pd = _dev(parents, torch.int32)
    acc = _dev(accepted, torch.int32)
    new = lib.conv_commit(acc, xd, pd, _dev(state))
    assert np.abs(new.cpu().numpy() - ref).max() == 0.0          # copies only
    s = _dev(state)
    lib.conv_commit(acc, xd, pd, s, out=s)
    assert torch.equal(s, new)


def test_conv_errors_reported(lib):
    B, T, C, K = 2, 16, 32, 4
    parents, x, state, w, bias = _case(T, "random", B, C, K, False)
    bad = parents.copy()
    bad[1, 5] = 9                                            # parent after its child
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.tree_conv(_dev(x), _dev(state), _dev(w), _dev(bad, torch.int32), bias=_dev(bias), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x1
    fixed = bad.copy()
    fixed[1, 5] = 0                                          # read as the sanitised tree
    ref = oracle.tree_conv_batch(fixed, x, state, w, bias, "silu")
    y = lib.tree_conv(_dev(x), _dev(state), _dev(w), _dev(bad, torch.int32), bias=_dev(bias))
    assert rel_err(y.cpu().numpy(), ref) <= 1e-5
    err.zero_()
    acc = torch.tensor([T, -3], dtype=torch.int32, device="cuda")
    new = lib.conv_commit(acc, _dev(x), _dev(parents, torch.int32), _dev(state), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x4
    assert torch.equal(new, _dev(state))                     # nothing accepted
