"""A bounded device wait that runs out, on the GPU.

Every pipeline wait in the kernels (mbarriers and the fused decode kernel's
cross-CTA ready counters) gives up after a time limit, sets MOE_DEV_TIMEOUT,
lets the kernel's own copies and MMAs land, frees its tensor memory and exits.
Here the limit is cut to a few nanoseconds so that the waits run out on three
paths: the 128-row grouped GEMM (with the tensor-core router), the fused
decode kernel (with the fused route kernel) and the ring combine. The call must come back with
MOE_ERR_TIMEOUT, nothing faults or hangs, and after the limit is restored the
next call is exact against the oracle on the same device context.
"""
import numpy as np
import pytest
import torch

import synth
from expert_moe_layer_gb300 import binding as B
from gpu_cases import DeviceCase, check_forward

pytestmark = pytest.mark.gpu

W = synth.Workload
CASES = {
    # 128-token tiles, K = 2048 per unit: each epilogue and MMA wait lasts
    # microseconds
    "gemm_tc": W("timeout_gemm_tc", T=600, H=2048, I=1024, E=8, K=2),
    # decode-sized: fused route kernel, gather, fused MLP (GEMM2 units wait on
    # the ready counters of other CTAs' GEMM1 units)
    "mlp_fused": W("timeout_mlp_fused", T=64, H=256, I=512, E=64, K=8, router_bias=True),
    # rows of 8 KB, four routed and two shared per token: the combine streams
    # them through its shared-memory ring (copier and reducer waits)
    "ring_combine": W("timeout_ring_combine", T=1024, H=4096, I=128, E=8, K=4, n_shared=2,
                      I_shared=128),
}


@pytest.mark.parametrize("name", list(CASES))
def test_wait_limit_runs_out_then_the_next_call_is_exact(name):
    c = DeviceCase(CASES[name])
    plan = B.forward_plan(c.cfg, c.wl.T)
    if name == "mlp_fused":
        assert plan.fused_mlp == 1 and plan.fused_route == 1
    elif name == "ring_combine":
        assert plan.fused_mlp == 0 and plan.fused_route == 0
    else:
        assert plan.fused_mlp == 0 and plan.cta_pairs == 0 and plan.tile_rows == 128
    try:
        B.set_wait_limit_ns(4)
        _, ws = c.forward()
        rc, flags = B.moe_get_status(ws)
        assert rc == 6 and flags & B.DEV_TIMEOUT, (rc, flags)
    finally:
        B.set_wait_limit_ns(0)
    torch.cuda.synchronize()
    check_forward(c)


def test_wait_limit_setter_restores_default():
    B.set_wait_limit_ns(123456789)
    B.set_wait_limit_ns(0)
    c = DeviceCase(CASES["mlp_fused"])
    check_forward(c)
