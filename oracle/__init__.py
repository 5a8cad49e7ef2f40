"""CPU oracle (test infrastructure only; never used by the product path)."""
from .oracle import *  # noqa: F401,F403
from .oracle import build_oracle, num_threads  # noqa: F401
