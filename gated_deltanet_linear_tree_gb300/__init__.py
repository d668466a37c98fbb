"""Closed-form tree verification for Gated DeltaNet layers on one GB300.

The compute lives in ``libcanopy.so`` (hand-written sm_103a CUDA, C ABI in
``include/canopy.h``); ``canopy`` is its thin Python binding and ``build``
compiles it in-tree with nvcc.
"""

from . import build  # noqa: F401
from . import canopy  # noqa: F401

__all__ = ["build", "canopy"]
