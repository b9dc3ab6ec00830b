"""CPU oracle of the Engram hot path.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline / reference legs of ``bench.py``.  Never by the
product package.
"""
from .engram_oracle import *  # noqa: F401,F403
