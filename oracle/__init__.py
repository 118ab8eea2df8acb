"""fp64 CPU oracle (test infrastructure only; see asp_oracle's header)."""
from .asp_oracle import *  # noqa: F401,F403
