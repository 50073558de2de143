"""GB300-native fused MoE layer forward (sm_103a CUDA kernels behind a C ABI).

``binding`` holds the ctypes wrappers of ``include/moe.h``. The kernels live
in ``csrc/`` and build in place into ``libmoe.so`` (see ``_build``).
"""
from . import binding  # noqa: F401
from .binding import (MoeConfig, MoeError, make_config, moe_align_permute,  # noqa: F401
                      moe_combine, moe_forward, moe_get_status, moe_grouped_mlp, moe_route)
