"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing ids, counts, offsets, the permutation and inv_pos must match
bit-exactly. Routing weights must agree within W_RTOL, and layer outputs per
element within |gpu - ref| <= 2e-2 + 2e-2*|ref|. Small layers are compared
element by element. The full-size layers are compared on all routing and
permutation arrays and on a sample of output tokens, run exactly as bench.py
runs them (moe_forward, one call).
"""
import numpy as np
import pytest
import torch

import synth
from expert_moe_layer_gb300 import binding as B
from oracle import moe_oracle as O

from gpu_cases import (ATOL, RTOL, W_ATOL, W_RTOL, DeviceCase, assert_close, check_forward,
                       sample_tokens, tile_edge_tokens, ws_views)

pytestmark = pytest.mark.gpu

W = synth.Workload
SMALL = {
    "tiny_f32": synth.TINY,
    "ragged_prefill": W("ragged_prefill", T=333, H=384, I=640, E=12, K=3),
    "ragged_decode": W("ragged_decode", T=77, H=256, I=384, E=16, K=4, router_bias=True),
    "grouped_shared": synth.DEEPSEEK.with_(name="grouped_shared", T=300, H=512, I=256,
                                           I_shared=384),
    "ep_rank1": synth.EP_SHARD.with_(name="ep_rank1", T=500, H=256, I=256),
    "f32_ragged": W("f32_ragged", T=90, H=256, I=384, E=6, K=2, act="f32", router="f32",
                    x_std=0.3),
    "k_equals_e": W("k_equals_e", T=40, H=128, I=128, E=8, K=8),
    "single_token": W("single_token", T=1, H=256, I=256, E=32, K=4, router_bias=True),
    # segments averaging >= 192 rows
    "wide_prefill": W("wide_prefill", T=1100, H=256, I=384, E=5, K=1),
    # long segments with enough work units: 256-token tiles on CTA pairs
    "pair_prefill": W("pair_prefill", T=4096, H=256, I=2048, E=8, K=2),
    # long segments with 256 to 511 units: 256-token tiles on single CTAs,
    # token rows gathered by GEMM1, GEMM2 overlapping it
    "single256": W("single256", T=2048, H=256, I=2048, E=8, K=2),
    # decode-sized segments with >= 152 GEMM1 units: both GEMMs in the fused
    # kernel (one tile per expert; then up to two ragged tiles per expert)
    "fused_decode": W("fused_decode", T=64, H=256, I=512, E=64, K=8, router_bias=True),
    "fused_two_tiles": W("fused_two_tiles", T=150, H=384, I=2048, E=16, K=4),
    # small batches route and align in one kernel: bf16 x with an fp32 router,
    # group-limited top-k with shared experts, an EP shard, and E > 256
    "f32_router_decode": W("f32_router_decode", T=16, H=256, I=256, E=8, K=2, router="f32"),
    "grouped_decode": synth.DEEPSEEK.with_(name="grouped_decode", T=24, H=256, I=256,
                                           I_shared=256),
    "ep_decode": synth.EP_SHARD.with_(name="ep_decode", T=32, H=256, I=256),
    # a few items over many local experts (24 items over 64)
    "ep_tiny": synth.EP_SHARD.with_(name="ep_tiny", T=3, H=256, I=256),
    "wide_router": W("wide_router", T=12, H=128, I=128, E=320, K=4, ep_size=2, ep_rank=1,
                     router_bias=True),
    # sigmoid scores with the selection-only score correction (e_score_correction_bias
    # reading), grouped, on each top-k path: the fused route kernel (T <= 128),
    # CTA per token (T < 256) and warp per token
    "sigmoid_select": W("sigmoid_select", T=40, H=256, I=256, E=64, K=6, n_group=8,
                        topk_group=4, rsf=2.5, n_shared=1, I_shared=256, router_bias=True,
                        bias_mode="select", scoring="sigmoid"),
    "sigmoid_select_mid": W("sigmoid_select_mid", T=200, H=256, I=256, E=64, K=6, n_group=8,
                            topk_group=4, rsf=2.5, router_bias=True, bias_mode="select",
                            scoring="sigmoid"),
    "sigmoid_select_wide": W("sigmoid_select_wide", T=300, H=256, I=256, E=32, K=4,
                             router_bias=True, bias_mode="select", scoring="sigmoid",
                             renormalize=False),
    # decode-sized batches on the fused route and MLP kernels: group-limited
    # sigmoid scores with the selection-only correction, no renormalisation,
    # rsf; a wide hidden size at 16 tokens
    "decode_grouped_select": W("decode_grouped_select", T=7, H=256, I=256, E=64, K=6,
                               n_group=8, topk_group=4, rsf=2.5, router_bias=True,
                               bias_mode="select", scoring="sigmoid", renormalize=False),
    "decode_wide_hidden": W("decode_wide_hidden", T=16, H=4096, I=384, E=16, K=4,
                            router_bias=True),
    # two shared experts over T >= 512 tokens: dense tiles on CTA pairs, ragged last tile
    "shared_pairs": W("shared_pairs", T=600, H=256, I=256, E=16, K=2, n_shared=2,
                      I_shared=384),
    # sigmoid with a logit bias, fp32 layer
    "sigmoid_f32": W("sigmoid_f32", T=50, H=128, I=128, E=8, K=2, act="f32", router="f32",
                     router_bias=True, scoring="sigmoid", x_std=0.3),
    # fp32 routers above 128 tokens run on CUDA cores: split over H for E <= 32
    # (bf16 x with a ragged last token batch; an fp32 layer whose last H slice
    # is half full, over two expert octets), one warp per expert beyond 32
    "f32_router_prefill": W("f32_router_prefill", T=701, H=512, I=256, E=8, K=2, router="f32"),
    "f32_layer_prefill": W("f32_layer_prefill", T=301, H=384, I=256, E=12, K=3, act="f32",
                           router="f32", x_std=0.3),
    "f32_router_wide": W("f32_router_wide", T=300, H=256, I=128, E=64, K=6, router="f32",
                         router_bias=True),
    # 128-token tiles with at least 152 GEMM1 units: GEMM2 overlaps GEMM1 and
    # takes each tile once GEMM1 has published it (one tile per expert, then
    # ragged segments of one or two tiles)
    "overlap_prefill": W("overlap_prefill", T=2048, H=256, I=384, E=64, K=2),
    "overlap_ragged": W("overlap_ragged", T=1500, H=384, I=512, E=40, K=3, router_bias=True),
    # more items than the single-CTA align takes: per-warp counts, then scan
    # and scatter in one pass (64 local experts), or the three passes (300)
    "align_fold": W("align_fold", T=1200, H=128, I=128, E=64, K=8),
    "align_three_pass": W("align_three_pass", T=640, H=128, I=128, E=300, K=16),
    # from 1024 tokens whose rows bring at least 48 KB each, the combine
    # streams them through a shared-memory ring: 8 KB rows, four routed and two
    # shared per token with rsf; an fp32 layer of six routed rows whose last
    # CTA takes fewer tokens
    "ring_shared": W("ring_shared", T=1024, H=4096, I=128, E=8, K=4, n_shared=2,
                     I_shared=128, rsf=2.5),
    "ring_f32": W("ring_f32", T=1030, H=2048, I=128, E=8, K=6, act="f32", router="f32",
                  x_std=0.3),
}
OVERLAP = ("overlap_prefill", "overlap_ragged")
# the combine streams their rows through the shared-memory ring
RING = ("ring_shared", "ring_f32")
SCORING = ("sigmoid_select", "sigmoid_select_mid", "sigmoid_select_wide", "sigmoid_f32")
FUSED = ("fused_decode", "fused_two_tiles", "grouped_shared")
ROUTE_FUSED = ("tiny_f32", "ragged_decode", "single_token", "f32_router_decode",
               "grouped_decode", "ep_decode", "ep_tiny", "wide_router", "decode_grouped_select",
               "decode_wide_hidden")
FULL = {
    "mixtral_prefill": synth.MIXTRAL,
    "deepseek_v2_prefill": synth.DEEPSEEK,
    "ep_shard": synth.EP_SHARD,
}

_cache = {}


def case(name):
    if name not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        wl = {**SMALL, **FULL}.get(name)
        if wl is None:
            T = int(name.split("_T")[1])
            wl = synth.QWEN_DECODE.with_(name=name, T=T)
        _cache[name] = DeviceCase(wl)
    return _cache[name]


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small(name):
    check_forward(case(name))


@pytest.mark.parametrize("T", synth.DECODE_TOKENS)
def test_forward_decode_full_shape(T):
    check_forward(case(f"qwen3_decode_T{T}"))


@pytest.mark.parametrize("name", list(FULL))
def test_forward_full_size_sampled(name):
    """Full-size layers, run as bench.py runs them: every routing and
    permutation array in full, and the output rows of 64 evenly spaced tokens
    plus every token that owns the first or last item of a GEMM tile (128-row
    steps inside each expert segment: the single-CTA tile, or each CTA's half
    of a 256-row pair tile), so that every tile of every segment has compared
    rows, its ragged end included."""
    c = case(name)
    plan = B.forward_plan(c.cfg, c.wl.T)
    step = min(plan.tile_rows, 128)
    edges = tile_edge_tokens(c, step)
    tokens = np.union1d(sample_tokens(c.wl.T), edges)
    counts, offsets, sorted_ids, _ = c.oracle_align(1)
    chosen = np.isin(np.arange(c.wl.T), tokens)
    for e in range(len(counts)):
        s, n = int(offsets[e]), int(counts[e])
        for r0 in range(s, s + n, step):
            rows = sorted_ids[r0:min(r0 + step, s + n)] // c.wl.K
            assert chosen[rows].any(), (name, e, r0)
    check_forward(c, tokens=tokens)


# ------------------------------------------------------------------ components
@pytest.mark.parametrize("name", ["ragged_prefill", "grouped_shared", "ragged_decode",
                                  "tiny_f32", "ep_rank1", *SCORING])
def test_route_entry_point(name):
    c = case(name)
    wl = c.wl
    ids = torch.empty(wl.T, wl.K, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, wl.K, dtype=torch.float32, device="cuda")
    ws = torch.empty(B.route_workspace_size(c.cfg, wl.T), dtype=torch.uint8, device="cuda")
    B.moe_route(c.cfg, wl.T, c.d["x"], c.d["router_w"], c.d["router_b"], ids, w, ws)
    assert B.moe_get_status(ws) == (0, 0)
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=W_RTOL, atol=W_ATOL)


def _align(c, ids_np, block, emap=None, cap=None):
    wl = c.wl
    El = wl.E_local
    cap = cap or B.align_cap(c.cfg, wl.T, block)
    ids = torch.from_numpy(ids_np).cuda()
    counts = torch.empty(El, dtype=torch.int32, device="cuda")
    offsets = torch.empty(El + 1, dtype=torch.int32, device="cuda")
    sorted_ids = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    inv_pos = torch.empty(wl.T * wl.K, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.align_workspace_size(c.cfg, wl.T), dtype=torch.uint8, device="cuda")
    em = None if emap is None else torch.from_numpy(emap).cuda()
    B.moe_align_permute(c.cfg, wl.T, ids, em, block, counts, offsets, sorted_ids, inv_pos,
                        cap, ws)
    st = B.moe_get_status(ws)
    return (counts.cpu().numpy(), offsets.cpu().numpy(), sorted_ids.cpu().numpy(),
            inv_pos.cpu().numpy(), st, cap)


@pytest.mark.parametrize("block", [1, 7, 16, 64, 128])
@pytest.mark.parametrize("name", ["ragged_prefill", "ep_rank1", "single_token", "ep_tiny",
                                  "wide_router", "align_fold", "align_three_pass"])
def test_align_entry_point(name, block):
    """The single-CTA per-warp counting sort (ragged_prefill, ep_rank1), the
    small-batch path of up to 64 items (single_token: 4 items; ep_tiny: 24
    items over 64 local experts; wide_router: 48 items of an EP shard with 160
    local experts), and the multi-CTA passes: per-CTA counts, then scan and scatter in
    one kernel (align_fold: 9600 items, 64 experts) or in two (align_three_pass:
    10240 items, 300 experts)."""
    c = case(name)
    counts, offsets, sorted_ids, inv_pos, st, cap = _align(c, c.ids, block)
    assert st == (0, 0)
    rc, ro, rs, ri = O.align_permute(c.ids, c.h["emap"], c.wl.E_local, block, cap)
    np.testing.assert_array_equal(counts, rc)
    np.testing.assert_array_equal(offsets, ro)
    np.testing.assert_array_equal(sorted_ids, rs)
    np.testing.assert_array_equal(inv_pos, ri)


@pytest.mark.parametrize("name", ["ep_rank1", "ep_tiny", "align_fold", "align_three_pass"])
def test_align_general_expert_map_and_bad_ids(name):
    """A permuted partial expert map, then flagged bad ids and map values, on
    the single-CTA align (ep_rank1: 4000 items), the small-batch one (ep_tiny:
    24 items) and the multi-CTA passes (align_fold, align_three_pass)."""
    c = case(name)
    wl = c.wl
    rng = np.random.default_rng(7)
    emap = np.full(wl.E, -1, dtype=np.int32)
    chosen = rng.choice(wl.E, wl.E_local, replace=False)
    emap[chosen] = rng.permutation(wl.E_local).astype(np.int32)
    counts, offsets, sorted_ids, inv_pos, st, cap = _align(c, c.ids, 16, emap)
    assert st == (0, 0)
    rc, ro, rs, ri = O.align_permute(c.ids, emap, wl.E_local, 16, cap)
    np.testing.assert_array_equal(sorted_ids, rs)
    np.testing.assert_array_equal(inv_pos, ri)
    # out-of-range ids and map values are dropped and flagged, never read
    ids = c.ids.copy()
    ids[0, 0] = wl.E + 5
    ids[1, 1] = -3
    emap2 = emap.copy()
    emap2[ids[2, 0]] = wl.E_local + 9
    _, _, sorted_ids, inv_pos, st, _ = _align(c, ids, 16, emap2)
    assert st[0] == 5 and st[1] & B.DEV_BAD_EXPERT_ID
    assert inv_pos[0] == -1 and inv_pos[1 * wl.K + 1] == -1 and inv_pos[2 * wl.K] == -1


@pytest.mark.parametrize("name", ["ragged_prefill", "ragged_decode", "f32_ragged",
                                  "grouped_shared", "fused_two_tiles"])
def test_grouped_mlp_and_combine_entry_points(name):
    c = case(name)
    wl = c.wl
    block = 16
    counts, offsets, sorted_ids, inv_pos = c.oracle_align(block)
    cap = len(sorted_ids)
    dt = c.d["x"].dtype
    y = torch.full((cap, wl.H), float("nan"), dtype=dt, device="cuda")
    ws = torch.empty(B.grouped_mlp_workspace_size(c.cfg, wl.T, cap), dtype=torch.uint8,
                     device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    B.moe_grouped_mlp(c.cfg, wl.T, c.d["x"], dev(sorted_ids), dev(counts), dev(offsets), cap,
                      c.d["w13"], c.d["w2"], y, ws)
    assert B.moe_get_status(ws) == (0, 0)
    rows = np.nonzero(sorted_ids < wl.T * wl.K)[0]
    ref = O.grouped_mlp(c.h["x"], sorted_ids, offsets, c.h["w13"], c.h["w2"], wl.K, rows)
    got = y.float().cpu().numpy()
    assert_close(got[rows], np.stack([ref[int(r)] for r in rows]), f"{name} y_perm")
    # combine from the oracle's y_perm rounded to the activation dtype
    yref = np.zeros((cap, wl.H), dtype=np.float32)
    for r in rows:
        yref[r] = ref[int(r)]
    y_dev = torch.from_numpy(yref).to(dt).cuda()
    shared = None
    if wl.n_shared:
        sh = sum(O.expert_mlp(c.h["x"], c.h["shared_w13"][s], c.h["shared_w2"][s])
                 for s in range(wl.n_shared))
        shared = torch.from_numpy(sh.astype(np.float32)).to(dt).cuda()
    out = torch.empty(wl.T, wl.H, dtype=dt, device="cuda")
    cws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    B.moe_combine(c.cfg, wl.T, y_dev, cap, dev(inv_pos), dev(c.w), shared, out, cws)
    assert B.moe_get_status(cws) == (0, 0)
    want = O.combine(y_dev.float().cpu().numpy(), inv_pos, c.w, wl.rsf,
                     None if shared is None else shared.float().cpu().numpy())
    assert_close(out.float().cpu().numpy(), want, f"{name} combine", atol=1e-2, rtol=1e-2)


@pytest.mark.parametrize("name", ["ragged_prefill", "ragged_decode"])
def test_grouped_mlp_drops_segments_outside_cap(name):
    """Caller-provided segments that start below 0 or run past cap are dropped
    and flagged (MOE_DEV_BAD_SEGMENT); the other experts' rows are still
    computed. ragged_prefill runs the 128-row grouped GEMM, ragged_decode the
    fused decode kernel."""
    c = case(name)
    wl = c.wl
    counts, offsets, sorted_ids, inv_pos = c.oracle_align(16)
    cap = len(sorted_ids)
    counts, offsets = counts.copy(), offsets.copy()
    El = wl.E_local
    bad = {0, 1, El - 1}                  # expert 0 now ends past expert 1's start
    offsets[1] = -5                       # starts before row 0
    counts[El - 1] = max(int(counts[El - 1]), 1) + 9
    offsets[El] = offsets[El - 1] + counts[El - 1]
    if offsets[El] <= cap:                # make the last segment run past cap
        offsets[El - 1] = cap - 2
        offsets[El] = cap - 2 + counts[El - 1]
    dt = c.d["x"].dtype
    y = torch.full((cap, wl.H), float("nan"), dtype=dt, device="cuda")
    ws = torch.empty(B.grouped_mlp_workspace_size(c.cfg, wl.T, cap), dtype=torch.uint8,
                     device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    B.moe_grouped_mlp(c.cfg, wl.T, c.d["x"], dev(sorted_ids), dev(counts), dev(offsets), cap,
                      c.d["w13"], c.d["w2"], y, ws)
    rc, flags = B.moe_get_status(ws)
    assert rc == 5 and flags & B.DEV_BAD_SEGMENT
    _, good_off, good_ids, _ = c.oracle_align(16)
    rows = [r for e in range(El) if e not in bad
            for r in range(int(good_off[e]), int(good_off[e]) + int(counts[e]))]
    rows = np.array([r for r in rows if good_ids[r] < wl.T * wl.K])
    ref = O.grouped_mlp(c.h["x"], good_ids, good_off, c.h["w13"], c.h["w2"], wl.K, rows)
    assert_close(y.float().cpu().numpy()[rows], np.stack([ref[int(r)] for r in rows]),
                 f"{name} y_perm of the valid segments")


# ------------------------------------------------------------------ edge cases
def test_no_local_items_gives_shared_only():
    c = case("grouped_shared")
    wl = c.wl
    d = c.d
    emap = torch.full((wl.E,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.workspace_size(c.cfg, wl.T), dtype=torch.uint8, device="cuda")
    out = torch.empty(wl.T, wl.H, dtype=d["x"].dtype, device="cuda")
    B.moe_forward(c.cfg, wl.T, d["x"], d["router_w"], None, d["w13"], d["w2"], d["shared_w13"],
                  d["shared_w2"], emap, out, ws)
    assert B.moe_get_status(ws) == (0, 0)
    sh = sum(O.expert_mlp(c.h["x"], c.h["shared_w13"][s], c.h["shared_w2"][s])
             for s in range(wl.n_shared))
    assert_close(out.float().cpu().numpy(), sh, "shared only")
    B.moe_forward(c.cfg, wl.T, d["x"], d["router_w"], None, d["w13"], d["w2"], None, None,
                  emap, out, ws)
    assert (out.float() == 0).all()


@pytest.mark.parametrize("fill", [0xFF, 0x7F])
@pytest.mark.parametrize("name", ["sigmoid_f32", "f32_ragged", "ragged_prefill", "overlap_prefill",
                                  "overlap_ragged", "align_fold", "fused_decode", "pair_prefill",
                                  "ep_rank1", "grouped_shared", "single256", "ring_shared"])
def test_forward_ignores_stale_workspace(name, fill):
    """moe_forward must not depend on what the workspace held before the call:
    every region it reads is written (or zeroed) by the call first. The
    workspace is filled with NaN bytes or huge finite values; the layer must
    still match the oracle on every path (fp32 with K split, 128-token tiles
    with GEMM2 overlapping GEMM1, the fused decode kernel, CTA pairs, an EP
    shard, shared experts, 256-token tiles on single CTAs, the ring combine)."""
    c = case(name)
    wl, d = c.wl, c.d
    ws = torch.full((B.workspace_size(c.cfg, wl.T),), fill, dtype=torch.uint8, device="cuda")
    out = torch.full((wl.T, wl.H), float("nan"), dtype=d["x"].dtype, device="cuda")
    B.moe_forward(c.cfg, wl.T, d["x"], d["router_w"], d["router_b"], d["w13"], d["w2"],
                  d["shared_w13"], d["shared_w2"], None, out, ws)
    assert B.moe_get_status(ws) == (0, 0)
    assert_close(out.float().cpu().numpy(), c.oracle_out(), f"{name} out, workspace {fill:#x}")


def test_zero_tokens_is_noop_and_repeat_calls_agree():
    c = case("ragged_decode")
    wl = c.wl
    d = c.d
    ws = torch.empty(B.workspace_size(c.cfg, wl.T), dtype=torch.uint8, device="cuda")
    out = torch.full((wl.T, wl.H), 3.0, dtype=d["x"].dtype, device="cuda")
    B.moe_forward(c.cfg, 0, d["x"], d["router_w"], None, d["w13"], d["w2"], None, None, None,
                  out, ws)
    torch.cuda.synchronize()
    assert (out.float() == 3.0).all()
    a, _ = c.forward()
    b, _ = c.forward()
    assert torch.equal(a, b)        # deterministic: no atomics in the reductions


def test_decode_repeat_calls_agree():
    """The decode-sized path (fused route and MLP kernels, split GEMM1 sums in
    a fixed order) gives the same bits on repeat calls."""
    c = case("decode_grouped_select")
    a, _ = c.forward()
    b, _ = c.forward()
    assert torch.equal(a, b)


def test_skewed_single_expert_segment():
    """Nearly all tokens choose expert 0 first: one long segment, many short or
    empty ones. (A much larger bias would leave the other experts' weights in
    exact ties near zero, which the tie-free inputs rule out.)"""
    wl = W("skewed", T=300, H=256, I=256, E=16, K=2, router_bias=True)
    c = DeviceCase(wl)
    c.h["router_b"] = c.h["router_b"].copy()
    c.h["router_b"][0] = 6.0
    c.d["router_b"] = torch.from_numpy(c.h["router_b"]).cuda()
    from oracle import cases
    x, _ = cases.gap_checked_x(wl, 0, c.h["router_w"], c.h["router_b"])
    c.h["x"] = x
    c.d["x"] = torch.from_numpy(x).to(torch.bfloat16).cuda()
    c.ids, c.w, c.p = O.route(x, c.h["router_w"], c.h["router_b"], top_k=2, renormalize=True)
    assert (c.ids[:, 0] == 0).mean() > 0.9
    check_forward(c)


@pytest.mark.parametrize("name", ["ragged_decode", "grouped_shared", "fused_decode",
                                  "decode_grouped_select"])
def test_forward_captured_in_cuda_graph_matches_eager(name):
    """moe_forward enqueues only stream work (no host sync, no allocation), so
    it can be captured once and replayed; replays must equal the eager call."""
    c = case(name)
    wl, d = c.wl, c.d
    eager, _ = c.forward()
    ws = torch.empty(B.workspace_size(c.cfg, wl.T), dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(eager)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        B.moe_forward(c.cfg, wl.T, d["x"], d["router_w"], d["router_b"], d["w13"], d["w2"],
                      d["shared_w13"], d["shared_w2"], None, out, ws, s)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert B.moe_get_status(ws) == (0, 0)


@pytest.mark.parametrize("name", ["pair_prefill", "ragged_prefill", *FUSED, *ROUTE_FUSED,
                                  *OVERLAP, *RING])
def test_plan_matches_the_kernels_launched(name):
    """moe_forward_plan (host only) names the path; moe_forward_timed counts
    the kernels that path launched. The fused cases must take the fused
    kernel, or their parity tests would not cover it."""
    c = case(name)
    wl, d = c.wl, c.d
    plan = B.forward_plan(c.cfg, wl.T)
    if name in FUSED:
        assert plan.fused_mlp == 1 and plan.tile_rows == 32
    if name in ROUTE_FUSED:
        assert plan.fused_route == 1
    if name in ("pair_prefill", "ragged_prefill"):
        assert plan.fused_route == 0 and plan.align_kernels == 1
    assert plan.gemm2_overlap == (1 if name in OVERLAP else 0)
    assert plan.combine_ring == (1 if name in RING else 0)
    ws = torch.empty(B.workspace_size(c.cfg, wl.T), dtype=torch.uint8, device="cuda")
    out = torch.empty(wl.T, wl.H, dtype=d["x"].dtype, device="cuda")
    n = B.moe_forward_timed(c.cfg, wl.T, d["x"], d["router_w"], d["router_b"], d["w13"],
                            d["w2"], d["shared_w13"], d["shared_w2"], None, out, ws,
                            [None] * 8)
    assert B.moe_get_status(ws) == (0, 0)
    assert n == plan.kernels
