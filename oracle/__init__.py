"""Float64 CPU oracle for dilution attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package; the CUDA library never does.
"""
from .dilution import *  # noqa: F401,F403
