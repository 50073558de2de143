"""Redundant experts (replica maps) on the GPU.

A layer of 16 logical experts over 2 ranks with 2 redundant replicas: each
rank holds 9 weight slots, experts 3 and 11 have a second replica on the other
rank (vLLM "physical" vs "logical" experts; num_redundant_experts). Item
(t, k) of an expert goes to replica t mod n_e of its n_e replicas (the reading
the oracle states). Each rank runs moe_forward with its replica map; the
routing, the permutation and the rank's partial output must match the oracle,
and the two partial outputs must add up to the unsharded layer.
"""
import numpy as np
import pytest
import torch

import synth
from expert_moe_layer_gb300 import binding as B
from gpu_cases import ATOL, RTOL, assert_close, sample_tokens, ws_views
from oracle import cases, moe_oracle as O

pytestmark = pytest.mark.gpu

E, K, H, I, EP, RED = 16, 4, 256, 256, 2, 2
PLACEMENT = [[(e // 8, e % 8)] for e in range(E)]
PLACEMENT[3] = [(0, 3), (1, 8)]
PLACEMENT[11] = [(1, 3), (0, 8)]
SLOTS = [list(range(8)) + [11], list(range(8, 16)) + [3]]   # logical expert of each slot


def _layer(T):
    wl = synth.Workload("replicas", T=T, H=H, I=I, E=E, K=K, router_bias=True)
    rw = synth.draw_tensor(wl, synth.ROUTER_W, 0)
    rb = synth.draw_tensor(wl, synth.ROUTER_B, 0)
    rb[[3, 11]] += 2.0                      # two hot experts
    x = cases.gap_checked_x(wl, 0, rw, rb)[0]
    w13 = synth.draw_tensor(wl, synth.W13, 0, local=False)
    w2 = synth.draw_tensor(wl, synth.W2, 0, local=False)
    return wl, x, rw, rb, w13, w2


def _cfg(rank):
    return B.make_config(E, K, H, I, True, ep_size=EP, ep_rank=rank, max_replicas=2,
                         num_redundant_experts=RED)


def _dev(a, bf16=True):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.to(torch.bfloat16) if bf16 else t).cuda()


@pytest.mark.parametrize("T", [5, 77, 2100])
def test_replica_ranks_match_oracle_and_sum_to_unsharded(T):
    # T=5: fused route kernel, small-batch align; T=77: fused route kernel;
    # T=2100: separate routing, 8400 items through the three-pass align
    wl, x, rw, rb, w13, w2 = _layer(T)
    maps = O.replica_maps(PLACEMENT, EP, 2)
    ids, w, _ = O.route(x, rw, rb, top_k=K, renormalize=True)
    tok = np.arange(T) if T <= 128 else sample_tokens(T, 48)
    total = np.zeros((tok.size, H))
    for r in range(EP):
        cfg = _cfg(r)
        pw13 = np.stack([w13[e] for e in SLOTS[r]])
        pw2 = np.stack([w2[e] for e in SLOTS[r]])
        ws = torch.empty(B.workspace_size(cfg, T), dtype=torch.uint8, device="cuda")
        out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        B.moe_forward(cfg, T, _dev(x), _dev(rw), _dev(rb, False), _dev(pw13), _dev(pw2),
                      None, None, torch.from_numpy(maps[r]).cuda(), out, ws)
        assert B.moe_get_status(ws) == (0, 0)
        v = ws_views(cfg, T, ws)
        np.testing.assert_array_equal(v["topk_ids"], ids)
        counts, offsets, sorted_ids, inv_pos = O.align_permute(ids, maps[r], 9, v["block_m"],
                                                               len(v["sorted_ids"]))
        np.testing.assert_array_equal(v["counts"], counts)
        np.testing.assert_array_equal(v["offsets"], offsets)
        np.testing.assert_array_equal(v["sorted_ids"], sorted_ids)
        np.testing.assert_array_equal(v["inv_pos"], inv_pos)
        ref = O.moe_forward(x, rw, pw13, pw2, top_k=K, renormalize=True, router_b=rb,
                            emap=maps[r], tokens=tok, routing=(ids, w))
        got = out.float().cpu().numpy()[tok]
        assert_close(got, ref, f"rank {r} partial output")
        total += got
    full = O.moe_forward(x, rw, w13, w2, top_k=K, renormalize=True, router_b=rb, tokens=tok,
                         routing=(ids, w))
    assert_close(total, full, "sum over ranks", atol=2 * ATOL, rtol=2 * RTOL)


def test_replica_map_without_replicas_is_flagged():
    wl, x, rw, rb, w13, w2 = _layer(40)
    maps = O.replica_maps(PLACEMENT, EP, 2)
    ids, w, _ = O.route(x, rw, rb, top_k=K, renormalize=True)
    bad = maps[0].copy()
    bad[5] = O.NO_REPLICA                   # expert 5 has no replica at all
    bad[6, 0] = 9                           # slot outside [0, 9)
    cfg = _cfg(0)
    n = 40 * K
    cap = int(B.align_cap(cfg, 40, 1))
    counts = torch.empty(9, dtype=torch.int32, device="cuda")
    offsets = torch.empty(10, dtype=torch.int32, device="cuda")
    sorted_ids = torch.empty(cap, dtype=torch.int32, device="cuda")
    inv_pos = torch.empty(n, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.align_workspace_size(cfg, 40), dtype=torch.uint8, device="cuda")
    B.moe_align_permute(cfg, 40, torch.from_numpy(ids).cuda(), torch.from_numpy(bad).cuda(), 1,
                        counts, offsets, sorted_ids, inv_pos, cap, ws)
    rc, flags = B.moe_get_status(ws)
    assert rc == 5 and flags & B.DEV_BAD_EXPERT_ID
    ip = inv_pos.cpu().numpy().reshape(40, K)
    assert (ip[(ids == 5) | (ids == 6)] == -1).all()
    good = (ids != 5) & (ids != 6)
    want = O.align_permute(np.where(good, ids, 0), maps[0], 9, 1, cap)[3].reshape(40, K)
    np.testing.assert_array_equal(ip[good] >= 0, want[good] >= 0)
