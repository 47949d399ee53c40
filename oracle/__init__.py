"""Oracle for the DFlash draft step, greedy verify-accept and draft-KV commit.

TEST INFRASTRUCTURE ONLY: a plain float64 CPU restatement of what the hot path
computes, written from the pages and pinned by tests/test_oracle_*.py against
closed forms, invariants, brute force and a toy greedy loop.  Only tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline leg may import it.  It
shares no code with the CUDA library and never imports it.
"""
from . import dflash_oracle  # noqa: F401
