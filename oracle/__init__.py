"""CPU oracle for the Ladder Transformer forward pass.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline / reference legs of ``bench.py``; never by the library.
"""
from .ladder_oracle import *  # noqa: F401,F403
