"""CPU float64 oracle (test infrastructure only; see cp_attention.py)."""
from .cp_attention import *  # noqa: F401,F403
