"""CPU float64 oracle for the MLA latent-KV hot path (test infrastructure only)."""
from .mla_oracle import *  # noqa: F401,F403
