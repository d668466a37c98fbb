"""fp64 CPU oracle for closed-form tree verification of Gated DeltaNet layers.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library and
imports nothing from it; the CUDA library does not import it.

Source of the method: the canopy page (projects.dotslasha.me/p/canopy.md),
sections "The gated delta rule", "The tree closed form" and "M1: Oracle and
tree generators".  Everything is computed in float64 on the float64 upcast of
the given input values.

Orientation.  The library's state is S of shape (dv, dk) and the rule is
    S_i = alpha_i * S_parent(i) (I - beta_i k_i k_i^T) + beta_i v_i k_i^T,
    o_i = S_i q_i,
which the page's "The gated delta rule" section names as the transpose of the
flash-linear-attention form (S of shape dk x dv, o = S^T q).  ``chain`` is
written in that other orientation on purpose, so the two cross-check.

Modules
  tree         ancestors, depths, masks and the DFS pre-order, written here
               (not shared)
  replay       the definition: the recurrence run along every root path
  chain        sequential recurrence for a chain, dk x dv orientation
  brute        every node's root path run as a fresh chain
  closed_form  log-space closed form with six solvers (dense, forward
               substitution, blocked forward substitution, Neumann, squaring,
               level-synchronous), fp64, plus an fp32 twin and the naive-ratio
               twin used by the stability pin; closed_form_heads carries
               every head of one stream at once (the round trip's check)
  commit       the accepted node's state from the pseudo-values
  conv         the tree-aware short causal convolution and its state commit

Pins (tests/test_oracle_*.py, run with -m "not gpu"): chain = sequential
recurrence; brute force on every tree of at most 8 nodes; closed form = replay
on 1,000 random trees for every solver; the T = 1 closed form; beta = 0, sibling,
homogeneity and relabelling invariants; nilpotency of G; commit = replay state
for every leaf; the page's printed figures (tests/golden/).
"""

from .tree import (  # noqa: F401
    validate_parent,
    root_path,
    depths,
    strict_ancestor_mask,
    cumulative_log_gate,
    dfs_preorder,
)
from .replay import replay, replay_batch  # noqa: F401
from .chain import chain_recurrence  # noqa: F401
from .brute import brute_force  # noqa: F401
from .closed_form import (  # noqa: F401
    closed_form,
    closed_form_batch,
    closed_form_heads,
    build_G_C,
    SOLVERS,
)
from .commit import commit, commit_batch  # noqa: F401
from .conv import tree_conv, tree_conv_batch, conv_commit, conv_commit_batch  # noqa: F401
