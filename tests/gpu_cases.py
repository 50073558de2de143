"""Shared helpers of the GPU parity tests and smoke(): device copies of a
gap-checked case, and the comparison rules.

Inputs come only from ``synth`` (through ``oracle.cases`` for the tie-free
token rows). Expected values come only from ``oracle``. Weights of large
layers are kept on the host as bf16 bit patterns and widened one expert at a
time when the oracle needs them.
"""
from __future__ import annotations

import numpy as np
import torch

import synth
from expert_moe_layer_gb300 import binding as B
from oracle import cases, moe_oracle as O

# Output tolerance per element for bf16 and tf32 paths:
#   |gpu - ref| <= ATOL + RTOL * |ref|
ATOL, RTOL = 2e-2, 2e-2
# Routing weights: the GPU's fp32 logits differ from the oracle's
# (fp64-summed then rounded) in summation order only, a few 1e-6 for the
# fan-ins used here, so the fp32 softmax probabilities agree to ~1e-5
# relative. 1e-4 leaves a 10x margin.
W_RTOL, W_ATOL = 1e-4, 1e-7


def cfg_of(wl) -> B.MoeConfig:
    return B.make_config(wl.E, wl.K, wl.H, wl.I, wl.renormalize, wl.n_group, wl.topk_group,
                         wl.rsf, wl.n_shared, wl.I_shared, wl.ep_size, wl.ep_rank, wl.act,
                         wl.router, wl.scoring, wl.bias_mode)


def _dev(a: np.ndarray, bf16: bool) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.to(torch.bfloat16) if bf16 else t.float()).cuda()


def _dev_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


class DeviceCase:
    """A gap-checked workload: host values for the oracle, device tensors for
    the library."""

    def __init__(self, wl, seed=0, lazy_weights=None):
        self.wl = wl
        bf = wl.act == "bf16"
        if lazy_weights is None:
            lazy_weights = bf and (wl.E_local * 3 * wl.H * wl.I > 64 * 2 ** 20)
        rw = synth.draw_tensor(wl, synth.ROUTER_W, seed)
        rb = synth.draw_tensor(wl, synth.ROUTER_B, seed) if wl.router_bias else None
        x, att = cases.gap_checked_x(wl, seed, rw, rb)
        self.h = dict(x=x, router_w=rw, router_b=rb, attempts=att,
                      emap=O.expert_map(wl.E, wl.ep_size, wl.ep_rank))
        if lazy_weights:
            e0 = wl.ep_rank * wl.E_local
            w13b = synth.draw_bf16_bits(seed, synth.W13, e0 * 2 * wl.I, wl.E_local * 2 * wl.I,
                                        wl.H, wl.std(synth.W13)).reshape(wl.E_local, 2 * wl.I, wl.H)
            w2b = synth.draw_bf16_bits(seed, synth.W2, e0 * wl.H, wl.E_local * wl.H, wl.I,
                                       wl.std(synth.W2)).reshape(wl.E_local, wl.H, wl.I)
            self.h["w13"], self.h["w2"] = synth.BF16Experts(w13b), synth.BF16Experts(w2b)
            self.d = dict(w13=_dev_bits(w13b), w2=_dev_bits(w2b))
        else:
            self.h["w13"] = synth.draw_tensor(wl, synth.W13, seed)
            self.h["w2"] = synth.draw_tensor(wl, synth.W2, seed)
            self.d = dict(w13=_dev(self.h["w13"], bf), w2=_dev(self.h["w2"], bf))
        self.h["shared_w13"] = self.h["shared_w2"] = None
        self.d["shared_w13"] = self.d["shared_w2"] = None
        if wl.n_shared:
            self.h["shared_w13"] = synth.draw_tensor(wl, synth.SHARED_W13, seed)
            self.h["shared_w2"] = synth.draw_tensor(wl, synth.SHARED_W2, seed)
            self.d["shared_w13"] = _dev(self.h["shared_w13"], bf)
            self.d["shared_w2"] = _dev(self.h["shared_w2"], bf)
        self.d["x"] = _dev(x, bf)
        self.d["router_w"] = _dev(rw, wl.router == "bf16")
        self.d["router_b"] = None if rb is None else torch.from_numpy(rb).cuda()
        ids, w, p = O.route(x, rw, rb, top_k=wl.K, renormalize=wl.renormalize,
                            n_group=wl.n_group, topk_group=wl.topk_group,
                            scoring=wl.scoring, bias_mode=wl.bias_mode)
        self.ids, self.w, self.p = ids, w, p
        self.cfg = cfg_of(wl)

    # ------------------------------------------------------------ oracle
    def oracle_out(self, tokens=None):
        wl, h = self.wl, self.h
        return O.moe_forward(h["x"], h["router_w"], h["w13"], h["w2"], top_k=wl.K,
                             renormalize=wl.renormalize, n_group=wl.n_group,
                             topk_group=wl.topk_group, rsf=wl.rsf, router_b=h["router_b"],
                             shared_w13=h["shared_w13"], shared_w2=h["shared_w2"],
                             emap=h["emap"], tokens=tokens, routing=(self.ids, self.w),
                             scoring=wl.scoring, bias_mode=wl.bias_mode)

    def oracle_align(self, block):
        return O.align_permute(self.ids, self.h["emap"], self.wl.E_local, block)

    # ------------------------------------------------------------ library
    def forward(self, with_shared=True, stream=None):
        wl, d = self.wl, self.d
        ws = torch.empty(B.workspace_size(self.cfg, wl.T), dtype=torch.uint8, device="cuda")
        out = torch.empty(wl.T, wl.H, dtype=d["x"].dtype, device="cuda")
        B.moe_forward(self.cfg, wl.T, d["x"], d["router_w"], d["router_b"], d["w13"], d["w2"],
                      d["shared_w13"] if with_shared else None,
                      d["shared_w2"] if with_shared else None, None, out, ws, stream)
        return out, ws


def ws_views(cfg, T, ws: torch.Tensor):
    """The routing / permutation arrays moe_forward leaves in its workspace."""
    lay = B.workspace_layout(cfg, T)
    K, El = cfg.top_k, (cfg.num_experts + cfg.num_redundant_experts) // cfg.ep_size

    def i32(off, n):
        return ws[off:off + 4 * n].view(torch.int32).cpu().numpy()

    return dict(topk_ids=i32(lay.topk_ids, T * K).reshape(T, K),
                topk_w=ws[lay.topk_w:lay.topk_w + 4 * T * K].view(torch.float32).cpu().numpy()
                .reshape(T, K),
                counts=i32(lay.counts, El), offsets=i32(lay.offsets, El + 1),
                sorted_ids=i32(lay.sorted_ids, lay.cap), inv_pos=i32(lay.inv_pos, T * K),
                block_m=lay.block_m)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str, atol=ATOL, rtol=RTOL):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite values"
    err = np.abs(gpu - ref)
    lim = atol + rtol * np.abs(ref)
    bad = err > lim
    if bad.any():
        i = np.unravel_index(np.argmax(err - lim), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu={gpu[i]} ref={ref[i]}")


def sample_tokens(T, n=64):
    if T <= n:
        return np.arange(T)
    return np.unique(np.linspace(0, T - 1, n).astype(np.int64))


def tile_edge_tokens(c: DeviceCase, tile_rows: int) -> np.ndarray:
    """Tokens that own the first and the last item of every tile of every
    expert segment, for tiles of tile_rows rows laid from each segment's start
    (the routed GEMMs' tile table on moe_forward's unpadded segments). A
    tile-table or out-of-bounds TMA mistake shows in exactly these rows: a
    segment's ragged last tile and the first tile after a segment boundary."""
    counts, offsets, sorted_ids, _ = c.oracle_align(1)
    K = c.wl.K
    toks = set()
    for e in range(len(counts)):
        s, n = int(offsets[e]), int(counts[e])
        for r0 in range(s, s + n, tile_rows):
            toks.add(int(sorted_ids[r0]) // K)
            toks.add(int(sorted_ids[min(r0 + tile_rows, s + n) - 1]) // K)
    return np.array(sorted(toks), dtype=np.int64)


def check_forward(c: DeviceCase, tokens=None):
    wl = c.wl
    out, ws = c.forward()
    rc, flags = B.moe_get_status(ws)
    assert rc == 0 and flags == 0, (rc, flags)
    v = ws_views(c.cfg, wl.T, ws)
    np.testing.assert_array_equal(v["topk_ids"], c.ids)
    np.testing.assert_allclose(v["topk_w"], c.w, rtol=W_RTOL, atol=W_ATOL)
    counts, offsets, sorted_ids, inv_pos = c.oracle_align(v["block_m"])
    np.testing.assert_array_equal(v["counts"], counts)
    np.testing.assert_array_equal(v["offsets"], offsets)
    np.testing.assert_array_equal(v["sorted_ids"], sorted_ids)
    np.testing.assert_array_equal(v["inv_pos"], inv_pos)
    tok = np.arange(wl.T) if tokens is None else tokens
    ref = c.oracle_out(tokens=tok)
    got = out[torch.from_numpy(tok).cuda()].float().cpu().numpy()
    assert_close(got, ref, f"{wl.name} out")
    return out, ws
