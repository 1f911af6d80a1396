"""CPU oracle for the MoE expert layer (test infrastructure; see moe_oracle)."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import __all__  # noqa: F401
