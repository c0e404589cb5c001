"""CPU oracle of the MuseSpark1x MoE decode block -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. The library never does.
"""
from .musemoe_oracle import *  # noqa: F401,F403
from .musemoe_oracle import Routing  # noqa: F401
