"""CPU oracle for the q4_0 weight-only int4 decode path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
legs may import this package.  The CUDA library never does, and this package
imports nothing from the CUDA library.  See :mod:`oracle.q4_oracle`.
"""
from .q4_oracle import *  # noqa: F401,F403
from . import q4_oracle  # noqa: F401
from . import q2_oracle  # noqa: F401
from . import q8_oracle  # noqa: F401
