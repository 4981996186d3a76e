"""CPU oracle for the QuaRot hot path (test infrastructure only).

Only the test-suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline import this package.  See ``quarot_oracle`` for the definitions.
"""
from .quarot_oracle import *  # noqa: F401,F403
from . import quarot_oracle  # noqa: F401
