"""CPU oracle for the lockstep multi-codebook frame decode.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg import this package. The CUDA product path never
does, and shares no code with it.
"""
from .orc import Oracle, build_oracle, lib  # noqa: F401
