"""CPU oracle for the W8A8 quantised MoE layer.

Test infrastructure only: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the CUDA library never does.
"""
from .oracle import *  # noqa: F401,F403
