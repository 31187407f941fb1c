"""fp64 CPU oracle of the routed int4 mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference arm
of ``bench.py`` may call it.  It shares no code with the CUDA path: it is plain
numpy written from the pages' definitions, with no blocking, fusion or
reordering beyond what those definitions state.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
closed forms, special cases, invariants or brute force on tiny inputs (see the
test docstrings).  Parity unpinned: none of the functions below.
"""
from .moe_oracle import *  # noqa: F401,F403
