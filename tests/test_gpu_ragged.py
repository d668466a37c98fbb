"""GPU parity of ragged batches: a per-stream tree length.

canopy page, "Design decisions", memory layout: the parent array plus a
per-sequence length for ragged batches.  Each stream b of a batch has its own
tree of lengths[b] nodes inside arrays of T rows.  Its outputs must be the
oracle's for that tree alone, whatever the rows past its length hold (here:
NaN q, k, v and beta, an invalid gate and out-of-range parents), and the rows
of o and of the workspace past its length must not be written.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import trees
from tests.gpu_helpers import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu

SENTINEL = 7.25


def _ragged_inputs(lengths, T, H, d, bf16, seed, fam="random"):
    """One tree per stream of its own length, padded to T rows with garbage."""
    B = len(lengths)
    rng = np.random.default_rng(seed)
    out = {"parent": np.full((B, T), 12345, np.int32),
           "q": np.full((B, T, H, d), np.nan, np.float32), "k": np.full((B, T, H, d), np.nan, np.float32),
           "v": np.full((B, T, H, d), np.nan, np.float32), "g": np.full((B, T, H), -1.0, np.float32),
           "beta": np.full((B, T, H), np.nan, np.float32), "S0": np.zeros((B, H, d, d), np.float32)}
    for b, L in enumerate(lengths):
        one = synth.make_inputs([trees.family(fam, max(L, 1), rng)], H, d, d, bf16, case=88, rnd=seed + b)
        for n in ("parent", "q", "k", "v", "g", "beta"):
            out[n][b, :L] = one[n][0, :L]
        out["S0"][b] = one["S0"][0]
    return out


def _to_device(inp, bf16):
    dt = torch.bfloat16 if bf16 else torch.float32
    d = {n: torch.from_numpy(inp[n]).to("cuda", dt).contiguous() for n in ("q", "k", "v")}
    for n in ("g", "beta", "S0"):
        d[n] = torch.from_numpy(inp[n]).cuda().contiguous()
    d["parent"] = torch.from_numpy(inp["parent"]).cuda().contiguous()
    return d


def _run(lib, lengths, T, H=2, d=128, bf16=True, seed=0, fam="random"):
    B = len(lengths)
    inp = _ragged_inputs(lengths, T, H, d, bf16, seed, fam)
    dev = _to_device(inp, bf16)
    ws = lib.workspace(B, T, H, d)
    views = lib.workspace_views(ws, B, T, H, d)
    views["u"].fill_(SENTINEL)
    views["l"].fill_(SENTINEL)
    views["depth"].fill_(-7)
    o = torch.full((B, T, H, d), SENTINEL, dtype=torch.float32, device="cuda")
    ln = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws, out=o,
               lengths=ln)
    err = lib.read_device_error(ws)
    return inp, dev, ws, views, o.cpu().numpy(), ln, err


def _check(inp, views, o, lengths, tol):
    worst = 0.0
    for b, L in enumerate(lengths):
        assert (o[b, L:] == SENTINEL).all(), b
        assert (views["u"][b, L:].cpu().numpy() == SENTINEL).all(), b
        assert (views["l"][b, L:].cpu().numpy() == SENTINEL).all(), b
        assert (views["depth"][b, L:].cpu().numpy() == -7).all(), b
        if L == 0:
            continue
        o_ref, _ = oracle.replay(inp["parent"][b, :L], inp["q"][b, :L], inp["k"][b, :L], inp["v"][b, :L],
                                 inp["g"][b, :L], inp["beta"][b, :L], inp["S0"][b], keep_states=False)
        assert np.isfinite(o[b, :L]).all(), b
        e = rel_err(o[b, :L], o_ref)
        worst = max(worst, e)
        assert e <= tol, (b, L, e)
        assert np.array_equal(views["depth"][b, :L].cpu().numpy(), oracle.depths(inp["parent"][b, :L])), b
    return worst


@pytest.mark.parametrize("T,lengths", [
    (256, [1, 2, 3, 17, 33, 63, 64, 65, 100, 127, 128, 129, 200, 255, 256, 0]),   # tensor cores, 64-node blocks
    (64, [0, 1, 5, 31, 32, 33, 63, 64]),                                           # the one-block kernel
    (3, [3, 1, 0, 2]),                                                             # the path replay (T <= 3)
])
def test_ragged_bf16_matches_each_streams_own_tree(lib, T, lengths):
    inp, dev, ws, views, o, ln, err = _run(lib, lengths, T)
    assert err == 0
    print(f"ragged T={T}: worst o err {_check(inp, views, o, lengths, TOL_BF16):.2e}")


@pytest.mark.parametrize("T,lengths", [(100, [100, 1, 0, 37, 64, 65]), (20, [20, 7, 1])])
def test_ragged_fp32_path(lib, T, lengths):
    inp, dev, ws, views, o, ln, err = _run(lib, lengths, T, bf16=False, seed=3)
    assert err == 0
    _check(inp, views, o, lengths, TOL_F32)


def test_ragged_chains_deep_blocks(lib):
    """Chains whose length ends inside a 64-node block, beyond the first."""
    lengths = [70, 129, 193, 256]
    inp, dev, ws, views, o, ln, err = _run(lib, lengths, 256, seed=5, fam="chain")
    assert err == 0
    _check(inp, views, o, lengths, TOL_BF16)


def test_ragged_commit(lib):
    """The commit after a ragged verify: each stream's accepted leaf gives the
    oracle's state; a stream with nothing accepted keeps S0; an accepted node
    at or past its stream's length is reported and keeps S0."""
    lengths = [150, 1, 64, 256, 90, 0]
    T, H = 256, 2
    inp, dev, ws, views, o, ln, err = _run(lib, lengths, T, H=H, seed=7)
    assert err == 0
    rng = np.random.default_rng(1)
    acc = [int(rng.choice(trees.leaves(inp["parent"][b, :L]))) if L else -1 for b, L in enumerate(lengths)]
    S = lib.commit(torch.tensor(acc, dtype=torch.int32, device="cuda"), dev["S0"], dev["k"], dev["parent"], ws,
                   lengths=ln)
    assert lib.read_device_error(ws) == 0
    S = S.cpu().numpy()
    for b, L in enumerate(lengths):
        if L == 0:
            assert np.array_equal(S[b], inp["S0"][b])
            continue
        path = oracle.root_path(inp["parent"][b, :L], acc[b])
        chain = np.arange(-1, len(path) - 1, dtype=np.int32)
        _, Sp = oracle.replay(chain, inp["q"][b][path], inp["k"][b][path], inp["v"][b][path], inp["g"][b][path],
                              inp["beta"][b][path], inp["S0"][b], keep_states=True)
        assert rel_err(S[b], Sp[-1]) <= TOL_BF16, b
    bad = list(acc)
    bad[0] = lengths[0]                                    # one past the stream's last node
    S2 = lib.commit(torch.tensor(bad, dtype=torch.int32, device="cuda"), dev["S0"], dev["k"], dev["parent"], ws,
                    lengths=ln)
    assert lib.read_device_error(ws) & 0x4
    assert np.array_equal(S2[0].cpu().numpy(), inp["S0"][0])


def test_lengths_at_T_equal_no_lengths(lib):
    """lengths[b] = T for every stream gives the same bits as no lengths."""
    for T in (40, 200):
        rng = np.random.default_rng(T)
        inp = synth.make_inputs([trees.family("random", T, rng) for _ in range(3)], 2, 128, 128, True, case=89)
        dev = _to_device(inp, True)
        ws = lib.workspace(3, T, 2, 128)
        o1 = lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws)
        ln = torch.full((3,), T, dtype=torch.int32, device="cuda")
        o2 = lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws,
                        lengths=ln)
        assert lib.read_device_error(ws) == 0
        assert torch.equal(o1, o2)


@pytest.mark.parametrize("T", [3, 64, 200])
def test_bad_length_is_reported(lib, T):
    lengths = [T, 2]
    inp = _ragged_inputs(lengths, T, 2, 128, True, 11)
    dev = _to_device(inp, True)
    ws = lib.workspace(2, T, 2, 128)
    for badlen in (-1, T + 5):
        ln = torch.tensor([T, badlen], dtype=torch.int32, device="cuda")
        lib.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws, lengths=ln)
        assert lib.read_device_error(ws) & 0x10
