"""Engram forward oracle -- TEST INFRASTRUCTURE ONLY.

A plain single-threaded fp64 CPU restatement of the Engram layer's forward
(the C source in ``engram_oracle.c``) and its numpy-facing wrappers.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA library.
"""
from .oracle import *  # noqa: F401,F403
