"""fp64 CPU oracle of the sparse-MLP decode path.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
benchmark's CPU-baseline leg.  The product path never imports it.
"""
from .decode import *  # noqa: F401,F403
from .decode import OracleDecoder, TokenRecord  # noqa: F401
