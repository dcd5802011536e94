"""fp64 CPU oracle of the NOSA decode step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package; the library never does.
"""
from .nosa_oracle import *  # noqa: F401,F403
