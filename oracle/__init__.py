"""fp64 CPU oracle (test infrastructure only; never called by the library)."""
from .scout_oracle import *  # noqa: F401,F403
from .scout_oracle import NEG_INF  # noqa: F401
