"""The dispatcher's cut-offs follow the measured table.

profiles/dispatch_H16_d128.jsonl holds, for every batch B in {1, 2, 4, 8, 16}
and tree size T in 1..8 (random trees, H = HV = 16, d = 128, bf16 inputs),
the median time of one verify call forced onto each path: the closed form on
the tensor cores and the path replay (one CTA per (stream, value head, node)
stepping the recurrence down the node's root path).  canopy page, "The tree
closed form": the closed form replaces the per-node replay; for a handful of
nodes the replay's single pass is cheaper than the closed form's fixed setup,
and this table says where.  The library's own answer (canopy_verify_plan, the
host query the entry point shares) must take the path the table says is
faster wherever the two differ by more than the run-to-run spread, and never
cost more than that spread over the faster one anywhere.
"""

import json
import os

import pytest

from gated_deltanet_linear_tree_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "profiles", "dispatch_H16_d128.jsonl")
BAND = 0.05     # medians closer than this are a tie (run-to-run spread of the table's p50s)


@pytest.fixture(scope="module")
def canopy():
    path = build.build()
    from gated_deltanet_linear_tree_gb300 import canopy as c
    c._lib = None
    c.load(path)
    return c


def cells():
    rows = [json.loads(line) for line in open(TABLE)]
    assert "env" in rows[0] and rows[0]["env"]["gpu"].startswith("NVIDIA GB300")
    rows = [r for r in rows if "B" in r]
    assert {(r["B"], r["T"]) for r in rows} == {(B, T) for B in (1, 2, 4, 8, 16) for T in range(1, 9)}
    return rows


def test_dispatch_follows_the_measured_table(canopy):
    clear = 0
    for r in cells():
        closed, replay = r["closed_form"]["p50"], r["path_replay"]["p50"]
        plan = canopy.verify_plan(r["T"], r["B"], r["H"], r["HV"], True, 128)
        assert plan in ("path_replay", "tc_block"), (r, plan)
        chosen = replay if plan == "path_replay" else closed
        assert chosen <= (1 + BAND) * min(closed, replay), (r, plan)
        if replay < (1 - BAND) * closed:
            assert plan == "path_replay", r
            clear += 1
        elif replay > (1 + BAND) * closed:
            assert plan == "tc_block", r
            clear += 1
    assert clear >= 30          # the table decides most cells outright


def test_forced_paths_are_the_two_the_table_timed(canopy):
    for r in cells():
        args = (r["T"], r["B"], r["H"], r["HV"], True, 128)
        assert canopy.verify_plan(*args, force="path_replay") == "path_replay"
        assert canopy.verify_plan(*args, force="closed_form") == "tc_block"
