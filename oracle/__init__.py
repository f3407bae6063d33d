"""fp64 CPU oracle of the MAPL boundary codec (test infrastructure only)."""
from .mapl_oracle import *  # noqa: F401,F403
