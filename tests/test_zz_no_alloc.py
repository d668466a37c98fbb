"""The allocation-free serial replay against the regular one.

canopy_serial_replay_static serves callers that cannot allocate device
memory (a host whose pool owns every allocation, or a loop that cannot pay
for cudaMalloc's synchronisation): its snapshots live in a fixed device array
inside the library.  Two calls in a row, with different trees, must each give
the output of canopy_serial_replay on the same inputs.  This file is
collected last so that a run that stops at the first failure has already run
everything else; it also passes when run alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth
from synth import trees
from tests.gpu_helpers import TOL_F32, oracle_outputs, rel_err, to_device

pytestmark = pytest.mark.gpu


def _case(seed, T, fam):
    rng = np.random.default_rng(seed)
    parents = [trees.family(fam, T, rng) for _ in range(1)]
    return synth.make_inputs(parents, 16, 128, 128, True, case=95, rnd=seed)


def test_static_serial_matches_regular_two_calls(lib):
    """Two calls in a row, different trees: each matches the regular replay
    and the fp64 oracle; the second call also runs without an err word (the
    library then keeps the bits in a spare word of its own array)."""
    for seed, T, fam, with_err in ((1, 16, "top4", True), (2, 31, "random", False)):
        inp = _case(seed, T, fam)
        dev = to_device(inp, True)
        err = torch.zeros(1, dtype=torch.int32, device="cuda") if with_err else None
        o_static = lib.serial_replay_static(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"],
                                            dev["parent"], err=err)
        ws = lib.workspace(1, T, 16, 128)
        o_ref = lib.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws)
        torch.cuda.synchronize()
        if with_err:
            assert int(err.item()) == 0
        assert rel_err(o_static.cpu().numpy(), o_ref.cpu().numpy()) <= TOL_F32
        o_orc, _ = oracle_outputs(inp)
        assert rel_err(o_static.cpu().numpy(), o_orc) <= TOL_F32


def test_static_serial_reports_a_bad_tree(lib):
    """A parent outside [0, i) is read as 0 (nothing is read out of bounds)
    and reported: CANOPY_DEVERR_TREE is OR-ed into the caller's zeroed err,
    and the output is the oracle's for the sanitised tree."""
    inp = _case(3, 20, "random")
    good = inp["parent"].copy()
    inp["parent"][0, 12] = 40
    dev = to_device(inp, True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = lib.serial_replay_static(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"],
                                 err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x1
    fixed = dict(inp, parent=good)
    fixed["parent"][0, 12] = 0
    o_orc, _ = oracle_outputs(fixed)
    assert rel_err(o.cpu().numpy(), o_orc) <= TOL_F32


def test_static_serial_rejects_sizes_beyond_its_array(lib):
    L = lib.load()
    p = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(9)]
    # 1 x 32 x 16 states of 128 x 128 fp32 = 32 MiB: over the limit, refused on the host
    st = L.canopy_serial_replay_static(p[0], p[1], p[2], 1, p[3], p[4], p[5], p[6], 32, 1, 16, 16, 128, 128,
                                       1.0, p[7], 0, None, None)
    assert st == 3
