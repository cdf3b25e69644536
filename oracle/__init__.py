"""CPU oracle for the CSA2 attention step -- test infrastructure only.

Importable by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py``; never by the library itself.
"""
from .oracle import *  # noqa: F401,F403
from .oracle import build, lib  # noqa: F401
