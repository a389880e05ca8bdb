"""CPU oracle (test infrastructure only; never imported by the library)."""
from .lynx_oracle import *  # noqa: F401,F403
