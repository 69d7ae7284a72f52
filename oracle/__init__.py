"""CPU oracle for the quantized paged KV decode path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU legs may import it.
"""
from .kvq_oracle import *  # noqa: F401,F403
from . import kvq_oracle  # noqa: F401
