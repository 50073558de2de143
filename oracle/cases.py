"""Gap-checked layer inputs for parity tests (test infrastructure only).

Bit-exact routing comparisons are only well posed when no top-k decision sits
on a near tie. This module draws a workload's inputs from ``synth``. It then
redraws any token row whose smallest routing decision gap, measured on the
oracle's fp32 selection scores, is below ``min_gap`` (1e-5). A redraw uses the row's
next attempt counter, so the final inputs are reproducible from
(seed, attempts). Only the token rows are redrawn; the weights are never
touched.
"""
from __future__ import annotations

import numpy as np

import synth
from .moe_oracle import expert_map, route, routing_min_gap

MIN_GAP = 1e-5


def gap_checked_x(wl, seed=0, router_w=None, router_b=None, min_gap=MIN_GAP,
                  max_rounds=64):
    """Token rows x[T, H] (float32) and their attempt counters."""
    if router_w is None:
        router_w = synth.draw_tensor(wl, synth.ROUTER_W, seed)
    if router_b is None and wl.router_bias:
        router_b = synth.draw_tensor(wl, synth.ROUTER_B, seed)
    attempts = np.zeros(wl.T, dtype=np.int32)
    x = synth.draw_tensor(wl, synth.X, seed, attempts)
    todo = np.arange(wl.T)
    for _ in range(max_rounds):
        _, _, sel = route(x[todo], router_w, router_b, top_k=wl.K,
                          renormalize=wl.renormalize, n_group=wl.n_group,
                          topk_group=wl.topk_group, scoring=wl.scoring,
                          bias_mode=wl.bias_mode)
        gap = routing_min_gap(sel, wl.K, wl.n_group, wl.topk_group)
        bad = todo[gap < min_gap]
        if bad.size == 0:
            return x, attempts
        for t in bad:
            attempts[t] += 1
            x[t] = synth.draw(seed, synth.X, int(t), 1, wl.H, wl.std(synth.X),
                              wl.act == "bf16",
                              attempts=attempts[t:t + 1])[0]
        todo = bad
    raise RuntimeError("could not draw tie-free token rows")


def build_case(wl, seed=0, min_gap=MIN_GAP, local=True):
    """Host inputs of a workload with tie-free routing, plus oracle routing."""
    d = synth.layer_inputs(wl, seed, local=local)
    d["x"], d["attempts"] = gap_checked_x(wl, seed, d["router_w"],
                                          d["router_b"], min_gap)
    d["emap"] = expert_map(wl.E, wl.ep_size, wl.ep_rank)
    ids, w, p = route(d["x"], d["router_w"], d["router_b"], top_k=wl.K,
                      renormalize=wl.renormalize, n_group=wl.n_group,
                      topk_group=wl.topk_group, scoring=wl.scoring,
                      bias_mode=wl.bias_mode)
    d["topk_ids"], d["topk_w"], d["p"] = ids, w, p
    d["wl"] = wl
    return d
