"""Seeded synthetic inputs for the tree-verify path.

This package draws draft trees (parent arrays) and the per-node activations
(q, k, v, gates, write strengths, committed state) with the shapes and value
distributions of the workloads described on the canopy page
(projects.dotslasha.me/p/canopy.md, "Design decisions" and "M1: Oracle and
tree generators").  It holds none of the method's arithmetic: it only makes
inputs.  Both the fp64 oracle (``oracle/``) and the CUDA path consume what it
returns; neither of them imports the other.
"""

from .trees import (  # noqa: F401
    chain,
    topk,
    schedule_tree,
    skewed,
    uniform_random,
    uniform_random_depth,
    relabel,
    dfs_preorder,
    level_order,
    tree_depth,
    node_depths,
    leaves,
    family,
)
from .values import make_inputs, make_aligned_inputs, round_bf16, stream_seed  # noqa: F401
from .configs import CONFIGS, config_inputs  # noqa: F401
