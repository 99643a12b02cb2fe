"""Float64 CPU oracle (test infrastructure only; never on the product path)."""
from .attention import *  # noqa: F401,F403
