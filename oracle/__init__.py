"""CPU oracle (test infrastructure only; never imported by the product path)."""
from .wq_oracle import *  # noqa: F401,F403
from .wq_oracle import GROUP  # noqa: F401
