"""fp64 CPU oracle (test infrastructure; see oracle/oracle.py for the scope rule)."""
from .oracle import *  # noqa: F401,F403
