"""Parity at the limits the host validation accepts.

- E = 512 experts with top_k = 32 (the kernel limits): 16 probabilities per
  lane in the warp top-k, 32 selection rounds, 512 local experts (more than
  the single-CTA align takes, so the three-pass align), on both top-k paths
  (CTA per token below 256 tokens, warp per token from 256).
- Group-limited top-k with the most groups (32 groups of 16, 8 kept).
- 1024 local weight slots (the E_local limit): 512 logical experts with 512
  redundant replicas on one rank, replica rows of 1, 2 and 16 entries (the
  max_replicas limit).
- T = 2^18 tokens (the token limit): with an fp32 router (the split-H router
  kernel, 2^19 items through the three-pass align, 256-token tiles on CTA
  pairs), and with top_k = 16 of 32 experts at H = 1024, where x_perm and
  y_perm hold 2^22 rows, 2^32 elements each, so row offsets past 2^31
  elements are used.

Routing and permutation arrays are compared whole and bit-exactly; outputs on
every token of the small cases and on sampled tokens at T = 2^18.
"""
import numpy as np
import pytest
import torch

import synth
from expert_moe_layer_gb300 import binding as B
from gpu_cases import DeviceCase, assert_close, check_forward, sample_tokens, ws_views
from oracle import cases, moe_oracle as O

pytestmark = pytest.mark.gpu

W = synth.Workload
MAX_T = 1 << 18

LIMITS = {
    "experts512_k32_cta_topk": W("experts512_k32_cta_topk", T=100, H=128, I=128, E=512, K=32,
                                 router_bias=True),
    "experts512_k32_warp_topk": W("experts512_k32_warp_topk", T=300, H=128, I=128, E=512,
                                  K=32, router_bias=True),
    "groups32": W("groups32", T=300, H=128, I=128, E=512, K=32, n_group=32, topk_group=8),
    # decode-sized batches at the limits: 16 tokens x 32 slots over 512
    # experts in the fused route kernel, and the most groups
    "decode_experts512_k32": W("decode_experts512_k32", T=16, H=128, I=128, E=512, K=32,
                               router_bias=True),
    "decode_groups32": W("decode_groups32", T=16, H=128, I=128, E=512, K=32, n_group=32,
                         topk_group=8),
}


@pytest.mark.parametrize("name", list(LIMITS))
def test_expert_and_top_k_limits(name):
    check_forward(DeviceCase(LIMITS[name]))


@pytest.mark.parametrize("wl", [
    W("max_tokens_f32_router", T=MAX_T, H=128, I=128, E=8, K=2, router="f32"),
    W("max_tokens_wide_rows", T=MAX_T, H=1024, I=128, E=32, K=16),
], ids=lambda wl: wl.name)
def test_token_limit(wl):
    check_forward(DeviceCase(wl), tokens=sample_tokens(wl.T, 48))


# 1024 local slots: slot e holds logical expert e; expert 0 has 15 more
# replicas (slots 512..526), experts 1..497 one more each (slots 527..1023).
E_LOG, E_SLOTS, R_MAX = 512, 1024, 16


def _placement():
    placement = [[(0, e)] for e in range(E_LOG)]
    placement[0] += [(0, 512 + j) for j in range(15)]
    for e in range(1, 498):
        placement[e].append((0, 526 + e))
    slots = np.empty(E_SLOTS, np.int64)
    for e, reps in enumerate(placement):
        for _, s in reps:
            slots[s] = e
    return placement, slots


def test_local_slot_limit_with_replicas():
    T, K, H, I = 300, 8, 128, 128
    wl = W("slots1024", T=T, H=H, I=I, E=E_LOG, K=K, router_bias=True)
    rw = synth.draw_tensor(wl, synth.ROUTER_W, 0)
    rb = synth.draw_tensor(wl, synth.ROUTER_B, 0)
    rb[0] += 3.0                                   # a hot expert over its 16 replicas
    x = cases.gap_checked_x(wl, 0, rw, rb)[0]
    w13 = synth.draw_tensor(wl, synth.W13, 0, local=False)
    w2 = synth.draw_tensor(wl, synth.W2, 0, local=False)
    placement, slots = _placement()
    emap = O.replica_maps(placement, 1, R_MAX)[0]
    assert emap.shape == (E_LOG, R_MAX)
    pw13, pw2 = w13[slots], w2[slots]
    cfg = B.make_config(E_LOG, K, H, I, True, max_replicas=R_MAX,
                        num_redundant_experts=E_SLOTS - E_LOG)
    assert B.validate_config(cfg) == 0

    def dev(a, bf16=True):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.to(torch.bfloat16) if bf16 else t).cuda()

    ws = torch.empty(B.workspace_size(cfg, T), dtype=torch.uint8, device="cuda")
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    B.moe_forward(cfg, T, dev(x), dev(rw), dev(rb, False), dev(pw13), dev(pw2), None, None,
                  torch.from_numpy(emap).cuda(), out, ws)
    assert B.moe_get_status(ws) == (0, 0)
    ids, w, _ = O.route(x, rw, rb, top_k=K, renormalize=True)
    v = ws_views(cfg, T, ws)
    np.testing.assert_array_equal(v["topk_ids"], ids)
    counts, offsets, sorted_ids, inv_pos = O.align_permute(ids, emap, E_SLOTS, v["block_m"],
                                                           len(v["sorted_ids"]))
    np.testing.assert_array_equal(v["counts"], counts)
    np.testing.assert_array_equal(v["offsets"], offsets)
    np.testing.assert_array_equal(v["sorted_ids"], sorted_ids)
    np.testing.assert_array_equal(v["inv_pos"], inv_pos)
    assert (counts[512:527] > 0).all()             # all 16 replicas of expert 0 in use
    ref = O.moe_forward(x, rw, pw13, pw2, top_k=K, renormalize=True, router_b=rb, emap=emap,
                        routing=(ids, w))
    assert_close(out.float().cpu().numpy(), ref, "1024 slots")
    # identical weights in every replica: the layer equals the plain one
    full = O.moe_forward(x, rw, w13, w2, top_k=K, renormalize=True, router_b=rb,
                         routing=(ids, w))
    assert_close(out.float().cpu().numpy(), full, "1024 slots vs unsharded")
