"""fp64 CPU oracle for causal sliding-window attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use it.
"""
from .swa_oracle import *  # noqa: F401,F403
