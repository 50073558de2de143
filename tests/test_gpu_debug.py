"""The bounds-checked build, libmoe_debug.so, on the small parity cases.

Its kernels also check the indices they derive themselves and trust in
libmoe.so: tile-table entries against the tile table and the permuted
buffers, output rows and columns, weight rows, the sorted positions the
gather and the combine read, and the top-k ids. It stands in for a memory
checker. Here it runs

- its self-test: one check fails in a kernel that touches no memory, and the
  record (count, site, index, bound) arrives and is cleared by the read;
- every small forward case of the parity tests, compared with the oracle as
  there and bit for bit with libmoe.so on the same inputs;
- the parity tests of the separate entry points (route, align, grouped MLP
  and combine, dropped segments, expert-parallel dispatch / compute /
  combine with and without replicas, the expert and top-k limits) through
  the debug library;

and after each one no check may have failed.
"""
import pytest
import torch

import test_gpu_ep as EP
import test_gpu_limits as LIM
import test_gpu_parity as P
from expert_moe_layer_gb300 import binding as B
from gpu_cases import DeviceCase, check_forward

pytestmark = pytest.mark.gpu


def _clean(rec, what):
    assert rec.count == 0, (f"{what}: {rec.count} failed bounds checks; first at "
                            f"{B.debug_site(rec.site)}, index {rec.index}, bound {rec.bound}")


def test_selftest_record_arrives_and_is_cleared():
    with B.debug_library():
        assert B.debug_build()
        B.debug_take()
        B.debug_selftest()
        rec = B.debug_take()
        assert rec.count == 1
        assert rec.site >> 16 == 1  # moe_api.cu
        assert (rec.index, rec.bound) == (5, 4)
        _clean(B.debug_take(), "after the read")


@pytest.mark.parametrize("name", list(P.SMALL))
def test_forward_passes_every_check_and_matches_release(name):
    c = DeviceCase(P.SMALL[name])
    out_rel, _ = c.forward()
    with B.debug_library():
        B.debug_take()
        out_dbg, _ = check_forward(c)  # routing, permutation and outputs vs the oracle
        _clean(B.debug_take(), name)
    assert torch.equal(out_dbg, out_rel), f"{name}: debug and release outputs differ"


ENTRY = [
    (P.test_route_entry_point, ("ragged_prefill",)),
    (P.test_route_entry_point, ("grouped_shared",)),
    (P.test_route_entry_point, ("ragged_decode",)),
    (P.test_align_entry_point, ("ragged_prefill", 16)),
    (P.test_align_entry_point, ("ep_rank1", 1)),
    (P.test_align_entry_point, ("ep_tiny", 128)),
    (P.test_align_general_expert_map_and_bad_ids, ("ep_rank1",)),
    (P.test_grouped_mlp_and_combine_entry_points, ("ragged_prefill",)),
    (P.test_grouped_mlp_and_combine_entry_points, ("ragged_decode",)),
    (P.test_grouped_mlp_and_combine_entry_points, ("f32_ragged",)),
    (P.test_grouped_mlp_and_combine_entry_points, ("grouped_shared",)),
    (P.test_grouped_mlp_and_combine_entry_points, ("fused_two_tiles",)),
    (P.test_grouped_mlp_drops_segments_outside_cap, ("ragged_prefill",)),
    (P.test_grouped_mlp_drops_segments_outside_cap, ("ragged_decode",)),
    (P.test_no_local_items_gives_shared_only, ()),
    (P.test_skewed_single_expert_segment, ()),
    (EP.test_ep_dispatch_exchange_compute_combine, ("ep4",)),
    (EP.test_ep_dispatch_exchange_compute_combine, ("ep2_sigmoid",)),
    (EP.test_ep_dispatch_to_replicas_exchange_compute_combine, ()),
    (EP.test_ep_dispatch_flags_bad_ids_and_handles_empty, ()),
    (LIM.test_expert_and_top_k_limits, ("experts512_k32_cta_topk",)),
    (LIM.test_expert_and_top_k_limits, ("groups32",)),
    (LIM.test_expert_and_top_k_limits, ("decode_experts512_k32",)),
]


@pytest.mark.parametrize("fn,args", ENTRY,
                         ids=[f"{fn.__name__}-{'-'.join(map(str, a))}" for fn, a in ENTRY])
def test_entry_point_parity_through_the_debug_library(fn, args):
    with B.debug_library():
        B.debug_take()
        fn(*args)
        _clean(B.debug_take(), fn.__name__)
