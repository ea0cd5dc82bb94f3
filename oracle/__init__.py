"""CPU oracle for the routed-expert W4A16 MoE layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this package: only the tests, the smoke check of ``__graft_entry__``
and the CPU-baseline leg of ``bench.py`` use it. It shares no code, constant or
helper with the CUDA library; the two meet only on the seeded inputs drawn by
``synth.py``.
"""
from .moe_oracle import *  # noqa: F401,F403
