"""fp64 CPU oracle for GrowPage's capacity-boundary engine.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline legs of bench.py, never by the product package.
"""

from .growpage import *  # noqa: F401,F403
