"""CPU oracle of the DSA hot path (test infrastructure; see dsa_oracle)."""
from .dsa_oracle import *  # noqa: F401,F403
