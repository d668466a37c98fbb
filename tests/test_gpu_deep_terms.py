"""GPU parity on inputs where the deep terms of the solve matter.

Every node of a stream shares one key (tests/deep_cases.py), so each term
(-G)^m R up to the tree's depth is visible in the output: a solve that drops
an ancestor or a round fails here, where with random keys it would pass.
Every solve is run: the fused tensor-core forward substitution and Neumann
kernels (one 64-node block), the blocked and level substitution beyond one
block, the squaring form and the split design.  Each output is compared with
the fp64 oracle replay at the bf16 tolerance and at the case's own bound
(ten times the error measured on GB300), and the state committed from the
same workspace is compared with the oracle's state of the committed node.
"""

import numpy as np
import pytest
import torch

from tests import deep_cases
from tests.gpu_helpers import TOL_BF16, oracle_outputs, page_metrics, rel_err, run_verify, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,solve", deep_cases.params())
def test_deep_terms(lib, name, solve):
    inp = deep_cases.inputs(name)
    o_ref, S_ref = oracle_outputs(inp, keep_states=True)
    dev = to_device(inp, bf16=True)
    o, ws, err = run_verify(lib, dev, solve=solve)
    assert err == 0
    on = o.cpu().numpy()
    assert np.isfinite(on).all()
    e = rel_err(on, o_ref)
    mabs, fro = page_metrics(on, o_ref)
    T = inp["parent"].shape[1]
    a = np.array([T - 1, int(np.flatnonzero(inp["parent"][1] == 0)[-1]) if T > 1 else 0], np.int32)
    Sn = lib.commit(torch.from_numpy(a).cuda(), dev["S0"], dev["k"], dev["parent"], ws)
    assert lib.read_device_error(ws) == 0
    es = rel_err(Sn.cpu().numpy(), S_ref[np.arange(2), a])
    print(f"DEEP {name} {solve} o_err {e:.3e} S_err {es:.3e} max_abs {mabs:.3e} rel_fro {fro:.3e}")
    assert e <= TOL_BF16 and es <= TOL_BF16
    bound = deep_cases.BOUND.get((name, solve))
    if bound is not None:
        assert bound <= TOL_BF16
        assert e <= bound, (name, solve, e, bound)
