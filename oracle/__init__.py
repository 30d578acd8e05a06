"""CPU oracle of the MoE FFN layer forward and backward (test infrastructure; see moe_oracle.py
and moe_backward.py).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg import this package.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
from . import moe_backward  # noqa: F401,E402
