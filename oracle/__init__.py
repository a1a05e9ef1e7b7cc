"""CPU oracle for the quantized MoE expert layer (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and reference
arms may import this package.  See moe_oracle.py for the definitions and the
readings of the pages they follow.
"""
from . import moe_oracle  # noqa: F401
