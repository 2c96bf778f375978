"""CPU oracle of the fused MoE layer forward -- test infrastructure only.

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
cpu_baseline / reference arm. It shares no code with the CUDA library.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import __all__  # noqa: F401
