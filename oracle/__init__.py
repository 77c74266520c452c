"""fp64 CPU oracle of the LaCT fast-weight chunk step: test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py (CPU baseline and the
reference arm) may import this package. The product path never does.
"""
from .lact_oracle import *  # noqa: F401,F403
