"""CPU float64 oracle (test infrastructure; see dcp_oracle.py)."""
from .dcp_oracle import *  # noqa: F401,F403
from . import dcp_oracle  # noqa: F401
