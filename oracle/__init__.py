"""CPU oracle for Gated DeltaNet tree verification (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library never calls it
and shares no code with it.
"""
from .gdn_oracle import *  # noqa: F401,F403
