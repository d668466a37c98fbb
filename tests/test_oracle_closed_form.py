"""The independent closed form against the replay on 1,000 random trees.

canopy page, "M1: Oracle and tree generators", acceptance criteria: every
solver within 1e-10 max-abs at d_k = d_v = 128 on trees of 1-256 nodes with
gates down to 0.01; the fp32 closed form within 1e-5 of the fp64 oracle.
"""

import numpy as np

import oracle
from oracle.closed_form import SOLVERS, build_G_C
from synth import trees

FAMILIES = ["random"] * 6 + ["chain", "top2", "top4", "skewed"]


def _case(rng, idx):
    T = int(rng.integers(1, 257))
    fam = FAMILIES[idx % len(FAMILIES)]
    p = trees.family(fam, T, rng)
    dk = dv = 128
    q = rng.standard_normal((T, 1, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, 1, dv))
    a = rng.uniform(0.01, 1.0, (T, 1))
    b = rng.uniform(0.0, 1.0, (T, 1))
    S0 = 0.1 * rng.standard_normal((1, dv, dk))
    return p, q, k, v, a, b, S0


def test_closed_form_matches_replay_1000_trees():
    rng = np.random.default_rng(20260801)
    worst = {s: 0.0 for s in SOLVERS}
    worst32 = (0.0, None)
    for idx in range(1000):
        p, q, k, v, a, b, S0 = _case(rng, idx)
        o, _ = oracle.replay(p, q, k, v, a, b, S0, keep_states=False)
        G, C, l, P = build_G_C(p, q[:, 0], k[:, 0], a[:, 0], b[:, 0])
        R = b[:, 0, None] * (v[:, 0] - P[:, None] * (k[:, 0] @ S0[0].T))
        base = P[:, None] * (q[:, 0] @ S0[0].T)
        for name, fn in SOLVERS.items():
            U = fn(G, R, p)
            err = np.abs(base + C @ U - o[:, 0]).max()
            worst[name] = max(worst[name], err)
            assert err <= 1e-10, (idx, name, len(p), err)
        if idx % 10 == 0:                     # the fp32 twin on every tenth tree
            O32, _, _ = oracle.closed_form(p, q[:, 0], k[:, 0], v[:, 0], a[:, 0], b[:, 0],
                                           S0[0], "fwdsub", np.float32)
            e32 = float(np.abs(O32 - o[:, 0]).max())
            if e32 > worst32[0]:
                worst32 = (e32, (idx, len(p)))
            assert e32 <= 1e-5, (idx, len(p), e32)
    print("worst fp64 per solver:", {k: f"{v:.2e}" for k, v in worst.items()},
          "worst fp32:", worst32)
