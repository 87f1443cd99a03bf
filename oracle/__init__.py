"""fp64 CPU oracle of the Stable LatentMoE layer.  TEST INFRASTRUCTURE:
imported only by the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs; the CUDA library never touches it."""
from .lmoe_oracle import *  # noqa: F401,F403
