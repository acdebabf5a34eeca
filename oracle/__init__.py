"""CPU oracle of the MoE stage1 + combine path.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  See moe_oracle.py.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import BLOCK, E4M3_MAX  # noqa: F401
