"""fp64 CPU oracle of the SpargeAttention2 hot path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs may import it.
"""
from .sa2_oracle import *  # noqa: F401,F403
from .sa2_oracle import RowSelection  # noqa: F401
