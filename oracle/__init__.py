"""CPU oracle of the fused MoE layer forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The CUDA library never does.
"""
from . import moe_oracle  # noqa: F401
