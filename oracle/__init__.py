"""fp64 CPU oracle of the sparse MoE layer forward.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the library. It shares no code with the
CUDA path. Every function is pinned by the CPU tests (invariants the pages
state, closed forms, brute force on tiny inputs and library special cases);
absolute parity with a trained checkpoint is not pinned (none is available).
"""
from .moe_oracle import *  # noqa: F401,F403
