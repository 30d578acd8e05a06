"""CPU oracle of the MoE FFN layer forward (test infrastructure; see moe_oracle.py).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg import this package.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
