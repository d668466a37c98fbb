"""The aligned-key GPU cases can see a truncated solve.

For every case of tests/deep_cases.py the planted mistakes a GPU solve could
make are built here on the CPU, from the oracle's own pieces, on exactly the
inputs the GPU test uses: forward substitution (or the split design's
inverse) that ignores ancestors more than two levels up, a Neumann series one
round short, a squaring form one factor short.  Each must miss the fp64
replay by more than the bound the GPU test holds that (case, solve) to, so a
GPU kernel with that mistake cannot pass.
"""

import math

import numpy as np
import pytest

import oracle
from oracle.closed_form import SOLVERS, build_G_C
from tests import deep_cases


def _planted(inp, solve):
    """o [B, T, H, dv] with the solve's planted mistake."""
    B, T, H, _ = inp["q"].shape
    out = np.zeros(inp["v"].shape)
    for b in range(B):
        p = inp["parent"][b]
        dep = oracle.depths(p)
        d = int(dep.max())
        for h in range(H):
            q, k, v = (inp[n][b, :, h].astype(np.float64) for n in ("q", "k", "v"))
            a, be = inp["g"][b, :, h].astype(np.float64), inp["beta"][b, :, h].astype(np.float64)
            S0 = inp["S0"][b, h].astype(np.float64)
            G, C, l, P = build_G_C(p, q, k, a, be)
            R = be[:, None] * (v - P[:, None] * (k @ S0.T))
            if solve in ("fwdsub", "split"):
                far = (dep[:, None] - dep[None, :]) > 2          # ancestors beyond the second dropped
                U = SOLVERS[solve](np.where(far, 0.0, G), R, p)
            elif solve == "neumann":
                Z, U = R.copy(), R.copy()
                for _ in range(d - 1):                           # one round short
                    Z = -(G @ Z)
                    U = U + Z
            else:
                nfac = math.ceil(math.log2(d + 1)) if d > 0 else 0
                U = R - G @ R if nfac >= 2 else R.copy()         # one factor short
                Gp = G
                for _ in range(1, nfac - 1):
                    Gp = Gp @ Gp
                    U = U + Gp @ U
            out[b, :, h] = P[:, None] * (q @ S0.T) + C @ U
    return out


@pytest.mark.parametrize("name,solve", deep_cases.params())
def test_planted_mistake_exceeds_the_gpu_bound(name, solve):
    inp = deep_cases.inputs(name)
    o_ref, _ = oracle.replay_batch(inp["parent"], inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["S0"])
    e = float(np.abs(_planted(inp, solve) - o_ref).max() / np.sqrt((o_ref ** 2).mean()))
    bound = deep_cases.BOUND[(name, solve)]
    assert e > bound, (name, solve, e, bound)
