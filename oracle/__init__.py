"""CPU oracle of the MoE-layer forward pass (test infrastructure only).

Imported by the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py``; never by the product library.
"""
from .smoe_oracle import *  # noqa: F401,F403
from . import smoe_oracle  # noqa: F401
