"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before any CUDA call."""
import ctypes

import pytest

from expert_moe_layer_gb300 import binding as B

MIX = dict(num_experts=8, top_k=2, hidden_size=4096, intermediate_size=14336)


def test_library_exports_every_header_function():
    L = B.lib()
    names = B.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/moe.h but not exported"
    assert set(names) == set(B._SIGS)


def test_debug_library_exports_every_header_function():
    L = B.lib(debug=True)
    for n in B.header_functions():
        assert hasattr(L, n), f"{n} declared in include/moe.h but not in libmoe_debug.so"
    # the build flag is a plain host function in both libraries
    assert L.moe_debug_build() == 1
    assert B.lib(debug=False).moe_debug_build() == 0


@pytest.mark.parametrize("debug", [False, True])
def test_only_the_header_functions_are_exported(debug):
    """Hidden visibility: two builds in one process (libmoe.so and
    libmoe_debug.so) must share no internal symbol. Template statics with
    default visibility become process-wide unique symbols, and one library's
    per-kernel set-up flags then skip the other's set-up."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    B.lib(debug=debug)
    from expert_moe_layer_gb300 import _build
    out = subprocess.run([nm, "-D", "--defined-only", _build.lib_path(debug)],
                         capture_output=True, text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if len(line.split()) >= 3}
    assert syms and syms <= set(B.header_functions()), sorted(syms - set(B.header_functions()))


def test_debug_entry_points_in_the_release_library_make_no_cuda_call():
    L = B.lib()
    rec = B.DebugRecord(count=7, site=9, index=3, bound=2)
    assert L.moe_debug_take(ctypes.byref(rec)) == 2  # MOE_ERR_UNSUPPORTED
    assert (rec.count, rec.site, rec.index, rec.bound) == (0, 0, 0, 0)
    assert L.moe_debug_take(None) == 1
    assert L.moe_debug_selftest(None) == 2
    assert ctypes.sizeof(B.DebugRecord) == 24
    assert isinstance(L.moe_last_cuda_error(), int)


def test_debug_library_switch_is_scoped():
    assert not B.debug_build()
    with B.debug_library():
        assert B.debug_build()
    assert not B.debug_build()
    assert B.debug_site((3 << 16) | 321) == "kernels_gemm_pair.cu:321"


def test_strerror_covers_all_codes():
    for code in range(7):
        assert B.strerror(code) and B.strerror(code) != "unknown status"
    assert B.strerror(99) == "unknown status"


def _cfg(**kw):
    base = dict(MIX)
    base.update(kw)
    return B.make_config(**base)


@pytest.mark.parametrize("kw,expect", [
    (dict(), 0),
    (dict(num_experts=160, top_k=6, hidden_size=5120, intermediate_size=1536,
          num_expert_group=8, topk_group=3, num_shared_experts=2,
          shared_intermediate_size=1536, routed_scaling_factor=16.0, renormalize=False), 0),
    (dict(num_experts=256, top_k=8, hidden_size=2048, intermediate_size=512, ep_size=4,
          ep_rank=1), 0),
    (dict(top_k=0), 1), (dict(top_k=9), 1),
    (dict(hidden_size=100), 1), (dict(intermediate_size=4000), 1),
    (dict(ep_size=3), 1),                 # E % ep_size != 0 (_ep_init assert)
    (dict(ep_size=4, ep_rank=4), 1), (dict(ep_size=4, ep_rank=-1), 1),
    (dict(num_expert_group=3, topk_group=1), 1),   # E % n_group
    (dict(num_expert_group=4, topk_group=5), 1),
    (dict(num_expert_group=4, topk_group=1, top_k=3), 1),  # K > kept experts
    (dict(num_shared_experts=1, shared_intermediate_size=0), 1),
    (dict(routed_scaling_factor=float("inf")), 1),
    (dict(num_experts=1024, top_k=2), 2),  # beyond kernel coverage
    (dict(num_experts=64, top_k=33), 2),
    (dict(num_experts=512, top_k=32), 0),  # at the kernel limits
    (dict(num_experts=512, top_k=32, num_expert_group=32, topk_group=8), 0),
    (dict(num_experts=512, top_k=2, num_expert_group=64, topk_group=8), 2),
    (dict(num_experts=512, top_k=2, max_replicas=16, num_redundant_experts=512), 0),
    (dict(num_experts=512, top_k=2, max_replicas=2, num_redundant_experts=513), 2),
    (dict(act_dtype="f32", router_dtype="bf16"), 2),
])
def test_validate_config(kw, expect):
    assert B.validate_config(_cfg(**kw)) == expect


def test_entry_points_reject_bad_args_without_cuda():
    cfg = _cfg()
    bad = _cfg(top_k=0)
    L = B.lib()
    null = None
    # invalid config -> INVALID_ARG before anything touches CUDA
    assert L.moe_forward(ctypes.byref(bad), 4, 16, 16, null, 16, 16, null, null, null, 16,
                         16, 1 << 30, null) == 1
    assert L.moe_route(ctypes.byref(cfg), -1, 16, 16, null, 16, 16, 16, 1 << 30, null) == 1
    # NULL / misaligned pointers
    assert L.moe_route(ctypes.byref(cfg), 4, null, 16, null, 16, 16, 16, 1 << 30, null) == 1
    assert L.moe_forward(ctypes.byref(cfg), 4, 18, 16, null, 16, 16, null, null, null, 16,
                         16, 1 << 30, null) == 1
    # workspace too small
    need = B.workspace_size(cfg, 4)
    assert need > 0
    assert L.moe_forward(ctypes.byref(cfg), 4, 16, 16, null, 16, 16, null, null, null, 16,
                         16, need - 1, null) == 3
    # cap below T*K + E_l*(block-1)
    assert L.moe_align_permute(ctypes.byref(cfg), 4, 16, null, 16, 16, 16, 16, 16,
                               int(B.align_cap(cfg, 4, 16)) - 1, 16, 1 << 30, null) == 3
    assert L.moe_align_permute(ctypes.byref(cfg), 4, 16, null, 0, 16, 16, 16, 16, 1000, 16,
                               1 << 30, null) == 1
    # T == 0 is a no-op
    assert L.moe_forward(ctypes.byref(cfg), 0, null, null, null, null, null, null, null,
                         null, null, null, 0, null) == 0
    # at most 2^18 tokens
    assert B.workspace_size(cfg, 1 << 18) > 0
    assert B.workspace_size(cfg, (1 << 18) + 1) == 0
    assert L.moe_forward(ctypes.byref(cfg), (1 << 18) + 1, 16, 16, null, 16, 16, null, null,
                         null, 16, 16, 1 << 40, null) == 1
    assert L.moe_route(ctypes.byref(cfg), (1 << 18) + 1, 16, 16, null, 16, 16, 16, 1 << 30,
                       null) == 1


def test_workspace_sizes_and_layout():
    cfg = _cfg()
    T = 4096
    assert B.align_cap(cfg, T, 16) == T * 2 + 8 * 15
    lay = B.workspace_layout(cfg, T)
    assert lay.total == B.workspace_size(cfg, T)
    assert lay.block_m == 1 and lay.cap == B.align_cap(cfg, T, lay.block_m) == T * 2
    offs = [lay.status, lay.topk_ids, lay.topk_w, lay.counts, lay.offsets, lay.sorted_ids,
            lay.inv_pos]
    assert all(o % 256 == 0 for o in offs) and len(set(offs)) == len(offs)
    assert B.route_workspace_size(cfg, T) >= 4 + 4 * T * 8
    assert B.align_workspace_size(cfg, T) > 0
    assert B.grouped_mlp_workspace_size(cfg, T, lay.cap) >= 2 * lay.cap * (4096 + 14336)
    assert B.workspace_size(_cfg(top_k=0), T) == 0


def _plan(wl, T=None):
    from gpu_cases import cfg_of
    return B.forward_plan(cfg_of(wl), wl.T if T is None else T)


def test_forward_plan_per_workload():
    import synth
    # Mixtral-shape prefill: bf16 routed GEMMs on CTA pairs, 256-token tiles,
    # fp32 router on CUDA cores split into 256-column slices of H
    p = _plan(synth.MIXTRAL)
    assert (p.tile_rows, p.cta_pairs, p.fused_mlp, p.gemm1_k_split) == (256, 1, 0, 1)
    assert p.gemm2_overlap == 0  # CTA pairs keep their own schedule
    assert (p.router_tensor_cores, p.router_partials) == (0, 4096 // 256)
    # route 2, align 1, gather + GEMM1 + GEMM2, combine
    assert p.kernels == 2 + 1 + 3 + 1
    assert p.fused_route == 0 and p.align_kernels == 1
    # decode: routing and align in one kernel; 32-token tiles; gather, GEMM1
    # and GEMM2 in the fused kernel; T=1 leaves few GEMM1 units, so GEMM1 is
    # also split over K (finished inside the fused kernel)
    for T in (8, 64):
        p = _plan(synth.QWEN_DECODE, T)
        assert (p.tile_rows, p.fused_mlp, p.gemm1_k_split, p.cta_pairs) == (32, 1, 1, 0)
        assert p.gemm2_overlap == 0
        assert (p.fused_route, p.align_kernels, p.router_partials) == (1, 0, 1)
        assert p.kernels == 1 + 2 + 1  # route+align, gather + fused MLP, combine
    p = _plan(synth.QWEN_DECODE, 1)
    assert (p.fused_mlp, p.tile_rows, p.fused_route) == (1, 32, 1) and p.gemm1_k_split > 1
    assert p.kernels == 1 + 2 + 1
    # the fused route kernel stops at 128 tokens
    assert _plan(synth.QWEN_DECODE, 128).fused_route == 1
    assert _plan(synth.QWEN_DECODE, 129).fused_route == 0
    # the one-pass scan and scatter stops where its per-CTA sums would read
    # more than 2^24 count entries: 2^19 items over 32 local experts take
    # three passes
    assert _plan(synth.Workload("fold_edge", T=1 << 18, H=128, I=128, E=32, K=2)).align_kernels == 3
    assert _plan(synth.Workload("fold_ok", T=1 << 15, H=128, I=128, E=32, K=2)).align_kernels == 2
    # DeepSeek-V2 shape: count, then scan and scatter in one pass (few
    # per-CTA counts); GEMM1 on single CTAs gathers its own token rows (no
    # gather kernel); shared experts add two GEMMs
    p = _plan(synth.DEEPSEEK)
    assert p.align_kernels == 2 and p.fused_mlp == 0 and p.fused_route == 0
    assert p.kernels == 2 + 2 + 2 + 2 + 1
    # single-CTA routed GEMMs over 128-token tiles, one K range: GEMM2
    # overlaps GEMM1
    assert (p.tile_rows, p.cta_pairs, p.gemm1_k_split, p.gemm2_overlap) == (128, 0, 1, 1)
    # EP shard: 256 rows per expert and 256 GEMM1 units on 256-token tiles,
    # under the 512 that CTA pairs take: 256-token tiles on single CTAs, GEMM2
    # overlapping GEMM1
    # six routed and two shared rows of 10 KB per token: the ring combine
    assert p.combine_ring == 1
    p = _plan(synth.EP_SHARD)
    assert (p.tile_rows, p.cta_pairs, p.gemm1_k_split, p.gemm2_overlap) == (256, 0, 1, 1)
    # two expected local rows of 4 KB per token: the register combine
    assert p.combine_ring == 0
    assert _plan(synth.MIXTRAL).combine_ring == 0
    assert _plan(synth.DEEPSEEK.with_(T=1023)).combine_ring == 0
    # 255 units on 256-token tiles: 128-token tiles
    assert _plan(synth.EP_SHARD.with_(T=8160)).tile_rows == 128
    # fp32 layers never take the bf16-only fused or pair kernels
    p = _plan(synth.TINY)
    assert (p.fused_mlp, p.cta_pairs, p.router_tensor_cores) == (0, 0, 0)
    # T = 0 launches nothing; bad configs are refused
    assert _plan(synth.TINY, 0).kernels == 0
    with pytest.raises(B.MoeError):
        B.forward_plan(_cfg(top_k=0), 16)


def test_replica_configs_are_validated_without_cuda():
    """Redundant experts: the replica map width, the redundant count and the
    divisibility of the physical experts are checked on the host; a replica
    config needs a map; the expert-parallel calls refuse replica maps."""
    L = B.lib()
    bp = ctypes.byref
    ok = _cfg(num_experts=16, top_k=4, hidden_size=256, intermediate_size=256, ep_size=2,
              max_replicas=2, num_redundant_experts=2)
    assert L.moe_validate_config(bp(ok)) == 0
    assert B.align_cap(ok, 4, 1) == 4 * 4        # 9 local slots, block 1: T*K rows
    for bad in (_cfg(max_replicas=17), _cfg(max_replicas=-1),
                _cfg(num_redundant_experts=2),  # redundant experts need a replica map
                _cfg(num_experts=16, ep_size=2, max_replicas=2, num_redundant_experts=1)):
        assert L.moe_validate_config(bp(bad)) == 1
    fake = 1 << 20
    # a replica config without a map
    assert L.moe_forward(bp(ok), 4, fake, fake, None, fake, fake, None, None, None, fake,
                         fake, 1 << 30, None) == 1
    assert L.moe_align_permute(bp(ok), 4, fake, None, 1, fake, fake, fake, fake, 1000, fake,
                               1 << 30, None) == 1
    # expert-parallel dispatch: the global placement map goes with replicas,
    # and only with them
    assert L.moe_ep_dispatch(bp(ok), 8, fake, fake, fake, None, *([fake] * 7), fake, 1 << 30,
                             None) == 1
    plain = _cfg(num_experts=16, top_k=4, hidden_size=256, intermediate_size=256, ep_size=2)
    assert L.moe_ep_dispatch(bp(plain), 8, fake, fake, fake, fake, *([fake] * 7), fake,
                             1 << 30, None) == 1


def test_ep_entry_points_reject_bad_args_without_cuda():
    cfg = _cfg(num_experts=16, top_k=4, hidden_size=256, intermediate_size=256, ep_size=4)
    L = B.lib()
    bp = ctypes.byref
    assert B.ep_dispatch_workspace_size(cfg, 64) > 0
    assert B.ep_expert_compute_workspace_size(cfg, 64) > 0
    assert B.ep_dispatch_workspace_size(_cfg(top_k=0), 64) == 0
    # dispatch: missing outputs, then a workspace that is too small
    assert L.moe_ep_dispatch(bp(cfg), 8, *([None] * 12), 0, None) == 1
    fake = 1 << 20
    args = [fake] * 3 + [None] + [fake] * 7      # no placement map: no replicas
    assert L.moe_ep_dispatch(bp(cfg), 8, *args, fake, 8, None) == 3
    # expert compute and combine: missing pointers
    assert L.moe_ep_expert_compute(bp(cfg), 8, *([None] * 7), 0, None) == 1
    assert L.moe_ep_combine(bp(cfg), 8, None, None, None, None, None, 0, None) == 1
    assert L.moe_ep_combine(bp(_cfg(top_k=0)), 8, None, None, None, None, None, 0, None) == 1


def test_binding_refuses_host_tensors_for_device_arguments():
    import torch
    assert B._p(None) is None and B._p(1 << 20) == 1 << 20
    with pytest.raises(ValueError, match="device tensors"):
        B._p(torch.zeros(4))
    with pytest.raises(ValueError, match="device tensors"):
        B.moe_combine(_cfg(), 4, torch.zeros(8, 4096), 8, torch.zeros(8, dtype=torch.int32),
                      torch.zeros(8), None, torch.zeros(4, 4096))
