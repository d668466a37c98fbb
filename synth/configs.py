"""The five workload cases, by what they are.

  0  tiny oracle case: B=1, H=2, dk=dv=32, T=8 uniform random tree, fp32 q/k/v
  1  Qwen3.5-9B-like GDN layer at batch 1: B=1, H=16, dk=dv=128, T=16 tree with
     branching schedule (4, 2, 1), bf16 q/k/v
  2  batched verify: B=16, H=16, dk=dv=128, T=64, one uniform random tree per
     stream with depth in [4, 20], bf16 q/k/v
  3  crossover sweep cell: B in {1,2,4,8,16}, T in {3,...,256}, family in
     {chain, top2..top8, skewed, random}, H=16, dk=dv=128, bf16 q/k/v
  4  verify/commit round trip: B=16, H=16, dk=dv=128, T=128 uniform random
     trees, 100 rounds, a fresh tree per round
"""

from __future__ import annotations

from . import trees
from .values import make_inputs, stream_seed

CONFIGS = {
    0: dict(B=1, H=2, dk=32, dv=32, T=8, bf16=False, tree="random"),
    1: dict(B=1, H=16, dk=128, dv=128, T=16, bf16=True, tree="schedule421"),
    2: dict(B=16, H=16, dk=128, dv=128, T=64, bf16=True, tree="random_depth_4_20"),
    3: dict(B=16, H=16, dk=128, dv=128, T=64, bf16=True, tree="random"),
    4: dict(B=16, H=16, dk=128, dv=128, T=128, bf16=True, tree="random"),
}

SWEEP_B = (1, 2, 4, 8, 16)
SWEEP_T = (3, 8, 16, 32, 64, 128, 256)
SWEEP_FAMILIES = ("chain", "top2", "top3", "top4", "top5", "top6", "top7", "top8",
                  "skewed", "random")


def make_tree(kind: str, T: int, rng):
    if kind == "schedule421":
        return trees.schedule_tree(T, (4, 2, 1))
    if kind == "random_depth_4_20":
        return trees.uniform_random_depth(T, rng, 4, 20)
    return trees.family(kind, T, rng)


def config_inputs(case: int, rnd: int = 0, **over):
    """Seeded inputs for a case; keyword overrides replace any field."""
    c = dict(CONFIGS[case])
    c.update(over)
    parents = [make_tree(c["tree"], c["T"], stream_seed(case, rnd, b)) for b in range(c["B"])]
    x = make_inputs(parents, c["H"], c["dk"], c["dv"], c["bf16"], case=case, rnd=rnd)
    x["cfg"] = c
    return x
