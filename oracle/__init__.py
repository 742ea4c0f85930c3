"""CPU oracle of the H3 DiT block: test infrastructure only (see h3_oracle.py)."""
from .h3_oracle import *  # noqa: F401,F403
