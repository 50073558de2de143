"""Expert-parallel dispatch and combine on the GPU, ranks simulated on one GPU.

ep_fused_moe_patch.py ``_ep_forward`` routes every rank's tokens globally,
sends each (token, slot) item to the rank that owns its expert, computes
there with top_k = 1, sends the weighted rows back and adds them up per
token. Here each rank is a separate set of calls on the same GPU, run one
after another:
- ``moe_route``, then ``moe_ep_dispatch`` on its own tokens;
- the exchange: the tests slice the send buffers in the order
  ``all_to_all_single`` would deliver them;
- ``moe_ep_expert_compute`` with the rank's expert shard;
- the reverse exchange, then ``moe_ep_combine``.

The dispatch buffers must equal the oracle's bit for bit (integer and copy
work). Expert rows and the final outputs are compared with the oracle's
unsharded layer within the bf16 tolerance.
"""
import numpy as np
import pytest
import torch

import synth
from expert_moe_layer_gb300 import binding as B
from gpu_cases import ATOL, RTOL, W_ATOL, W_RTOL, assert_close, cfg_of
from oracle import cases, moe_oracle as O

pytestmark = pytest.mark.gpu

W = synth.Workload
LAYERS = {
    # ep 4 with rsf and one shared expert; a rank without tokens
    "ep4": (W("ep4", T=1, H=256, I=256, E=16, K=4, rsf=1.5, n_shared=1, I_shared=256,
              ep_size=4), (37, 0, 64, 129)),
    # ep 2, grouped sigmoid routing with the selection correction, decode-sized
    "ep2_sigmoid": (W("ep2_sigmoid", T=1, H=256, I=512, E=32, K=6, n_group=4, topk_group=2,
                      router_bias=True, bias_mode="select", scoring="sigmoid", ep_size=2),
                    (5, 300)),
}


def _dev(a, bf16=True):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.to(torch.bfloat16) if bf16 else t.float()).cuda()


def _exchange(bufs, counts):
    """all_to_all_single over device tensors: rank d gets, in source-rank
    order, each source's rows for d."""
    ep = len(bufs)
    offs = [np.concatenate([[0], np.cumsum(c)]) for c in counts]
    return [torch.cat([bufs[s][int(offs[s][d]):int(offs[s][d + 1])] for s in range(ep)])
            for d in range(ep)]


@pytest.mark.parametrize("name", list(LAYERS))
def test_ep_dispatch_exchange_compute_combine(name):
    base, tokens = LAYERS[name]
    ep, E, K, H = base.ep_size, base.E, base.K, base.H
    El = E // ep
    full = base.with_(ep_size=1, ep_rank=0)
    rw = synth.draw_tensor(full, synth.ROUTER_W, 0)
    rb = synth.draw_tensor(full, synth.ROUTER_B, 0) if base.router_bias else None
    w13 = synth.draw_tensor(full, synth.W13, 0, local=False)
    w2 = synth.draw_tensor(full, synth.W2, 0, local=False)
    s13 = synth.draw_tensor(full, synth.SHARED_W13, 0) if base.n_shared else None
    s2 = synth.draw_tensor(full, synth.SHARED_W2, 0) if base.n_shared else None
    rkw = dict(top_k=K, renormalize=base.renormalize, n_group=base.n_group,
               topk_group=base.topk_group, scoring=base.scoring, bias_mode=base.bias_mode)
    cfg = [cfg_of(base.with_(ep_rank=r, T=max(t, 1))) for r, t in enumerate(tokens)]
    xs, sends, host_sends = [], [], []
    for r, T in enumerate(tokens):
        wl_r = base.with_(T=max(T, 1), ep_rank=r)
        x = cases.gap_checked_x(wl_r, 10 + r, rw, rb)[0][:T]
        xs.append(x)
        ids, w, _ = O.route(x, rw, rb, **rkw)
        host = O.ep_dispatch(x, ids, w, E, ep)
        host_sends.append(host)
        d_ids = torch.empty(T, K, dtype=torch.int32, device="cuda")
        d_w = torch.empty(T, K, dtype=torch.float32, device="cuda")
        d_x = _dev(x)
        if T:
            rws = torch.empty(B.route_workspace_size(cfg[r], T), dtype=torch.uint8,
                              device="cuda")
            B.moe_route(cfg[r], T, d_x, _dev(rw), None if rb is None else _dev(rb, False),
                        d_ids, d_w, rws)
            assert B.moe_get_status(rws) == (0, 0)
            np.testing.assert_array_equal(d_ids.cpu().numpy(), ids)
            np.testing.assert_allclose(d_w.cpu().numpy(), w, rtol=W_RTOL, atol=W_ATOL)
            d_ids = torch.from_numpy(ids).cuda()  # the oracle's weights feed the rest
            d_w = torch.from_numpy(w).cuda()
        n = T * K
        out = dict(counts=torch.full((ep,), -1, dtype=torch.int32, device="cuda"),
                   offsets=torch.full((ep + 1,), -1, dtype=torch.int32, device="cuda"),
                   pos=torch.full((n,), -7, dtype=torch.int32, device="cuda"),
                   x=torch.zeros(n, H, dtype=torch.bfloat16, device="cuda"),
                   ids=torch.full((n,), -7, dtype=torch.int32, device="cuda"),
                   w=torch.full((n,), -7.0, dtype=torch.float32, device="cuda"),
                   tok=torch.full((n,), -7, dtype=torch.int32, device="cuda"))
        ws = torch.empty(max(B.ep_dispatch_workspace_size(cfg[r], T), 16), dtype=torch.uint8,
                         device="cuda")
        B.moe_ep_dispatch(cfg[r], T, d_x, d_ids, d_w, out["counts"], out["offsets"], out["pos"],
                          out["x"], out["ids"], out["w"], out["tok"], ws)
        torch.cuda.synchronize()
        if T:
            assert B.moe_get_status(ws) == (0, 0)
        counts, pos, sx, sids, sw, stok = host
        np.testing.assert_array_equal(out["counts"].cpu().numpy(), counts)
        np.testing.assert_array_equal(out["offsets"].cpu().numpy(),
                                      np.concatenate([[0], np.cumsum(counts)]))
        np.testing.assert_array_equal(out["pos"].cpu().numpy(), pos)
        np.testing.assert_array_equal(out["ids"].cpu().numpy(), sids)
        np.testing.assert_array_equal(out["tok"].cpu().numpy(), stok)
        np.testing.assert_array_equal(out["w"].cpu().numpy(), sw)
        np.testing.assert_array_equal(out["x"].float().cpu().numpy(), sx.astype(np.float32))
        sends.append(out)

    counts = [h[0] for h in host_sends]
    recv = {k: _exchange([s[k] for s in sends], counts) for k in ("x", "ids", "w")}
    host_recv = {k: O.ep_exchange([h[i] for h in host_sends], counts)
                 for k, i in (("x", 2), ("ids", 3), ("w", 4))}
    ys = []
    for r in range(ep):
        R = recv["x"][r].shape[0]
        y = torch.zeros(R, H, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(max(B.ep_expert_compute_workspace_size(cfg[r], R), 16),
                         dtype=torch.uint8, device="cuda")
        B.moe_ep_expert_compute(cfg[r], R, recv["x"][r].contiguous(),
                                recv["ids"][r].contiguous(), recv["w"][r].contiguous(),
                                _dev(w13[r * El:(r + 1) * El]), _dev(w2[r * El:(r + 1) * El]),
                                y, ws)
        if R:
            assert B.moe_get_status(ws) == (0, 0)
            ref = O.ep_expert_compute(host_recv["x"][r], host_recv["ids"][r],
                                      host_recv["w"][r], w13[r * El:(r + 1) * El],
                                      w2[r * El:(r + 1) * El], r * El)
            assert_close(y.float().cpu().numpy(), ref, f"{name} rank {r} expert rows")
        ys.append(y)

    back = [[counts[s][r] for s in range(ep)] for r in range(ep)]
    rets = _exchange(ys, back)
    for r, T in enumerate(tokens):
        if T == 0:
            continue
        x = xs[r]
        sh = None
        d_sh = None
        if s13 is not None:
            sh = sum(O.expert_mlp(x, s13[s], s2[s]) for s in range(base.n_shared))
            d_sh = _dev(sh.astype(np.float32))
            sh = d_sh.float().cpu().numpy()  # the combine adds the bf16 shared output
        out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        cws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        B.moe_ep_combine(cfg[r], T, rets[r].contiguous(), sends[r]["pos"], d_sh, out, cws)
        assert B.moe_get_status(cws) == (0, 0)
        ref = O.moe_forward(x, rw, w13, w2, router_b=rb, rsf=base.rsf,
                            shared_w13=s13, shared_w2=s2, **rkw)
        assert_close(out.float().cpu().numpy(), ref, f"{name} rank {r} output")


# Redundant experts over 2 ranks (as in test_gpu_replicas): logical experts
# 0-15, experts 3 and 11 with a second replica; 9 weight slots per rank.
REP_E, REP_K, REP_H, REP_I, REP_EP, REP_SLOTS = 16, 4, 256, 256, 2, 9
REP_PLACEMENT = [[(e // 8, e % 8)] for e in range(REP_E)]
REP_PLACEMENT[3] = [(0, 3), (1, 8)]
REP_PLACEMENT[11] = [(1, 3), (0, 8)]
REP_SLOT_EXPERT = [list(range(8)) + [11], list(range(8, 16)) + [3]]


def test_ep_dispatch_to_replicas_exchange_compute_combine():
    """The token-dispatch form with redundant experts: each item goes to the
    rank of replica t mod n_e of its expert and carries the physical id; the
    send buffers equal the oracle's bit for bit, each rank computes its
    physical slots (a slot holds its logical expert's weights), and the
    combined outputs equal the unsharded layer."""
    base = W("ep_replicas", T=1, H=REP_H, I=REP_I, E=REP_E, K=REP_K, router_bias=True)
    rw = synth.draw_tensor(base, synth.ROUTER_W, 0)
    rb = synth.draw_tensor(base, synth.ROUTER_B, 0)
    rb[[3, 11]] += 2.0                                  # two hot experts
    w13 = synth.draw_tensor(base, synth.W13, 0, local=False)
    w2 = synth.draw_tensor(base, synth.W2, 0, local=False)
    pmap = O.physical_map(REP_PLACEMENT, REP_EP, REP_SLOTS, 2)
    d_pmap = torch.from_numpy(pmap).cuda()
    tokens = (70, 41)
    cfg = [B.make_config(REP_E, REP_K, REP_H, REP_I, True, ep_size=REP_EP, ep_rank=r,
                         max_replicas=2, num_redundant_experts=2) for r in range(REP_EP)]
    xs, sends, host_sends = [], [], []
    for r, T in enumerate(tokens):
        x = cases.gap_checked_x(base.with_(T=T), 30 + r, rw, rb)[0]
        xs.append(x)
        ids, w, _ = O.route(x, rw, rb, top_k=REP_K, renormalize=True)
        assert (ids == 3).any() and (ids == 11).any()
        host = O.ep_dispatch(x, ids, w, REP_E, REP_EP, pmap, REP_SLOTS)
        host_sends.append(host)
        n = T * REP_K
        out = dict(counts=torch.full((REP_EP,), -1, dtype=torch.int32, device="cuda"),
                   offsets=torch.full((REP_EP + 1,), -1, dtype=torch.int32, device="cuda"),
                   pos=torch.full((n,), -7, dtype=torch.int32, device="cuda"),
                   x=torch.zeros(n, REP_H, dtype=torch.bfloat16, device="cuda"),
                   ids=torch.full((n,), -7, dtype=torch.int32, device="cuda"),
                   w=torch.full((n,), -7.0, dtype=torch.float32, device="cuda"),
                   tok=torch.full((n,), -7, dtype=torch.int32, device="cuda"))
        ws = torch.empty(B.ep_dispatch_workspace_size(cfg[r], T), dtype=torch.uint8,
                         device="cuda")
        B.moe_ep_dispatch(cfg[r], T, _dev(x), torch.from_numpy(ids).cuda(),
                          torch.from_numpy(w).cuda(), out["counts"], out["offsets"], out["pos"],
                          out["x"], out["ids"], out["w"], out["tok"], ws, phys_map=d_pmap)
        assert B.moe_get_status(ws) == (0, 0)
        counts, pos, sx, sids, sw, stok = host
        np.testing.assert_array_equal(out["counts"].cpu().numpy(), counts)
        np.testing.assert_array_equal(out["pos"].cpu().numpy(), pos)
        np.testing.assert_array_equal(out["ids"].cpu().numpy(), sids)
        np.testing.assert_array_equal(out["tok"].cpu().numpy(), stok)
        np.testing.assert_array_equal(out["w"].cpu().numpy(), sw)
        np.testing.assert_array_equal(out["x"].float().cpu().numpy(), sx.astype(np.float32))
        sends.append(out)

    counts = [h[0] for h in host_sends]
    recv = {k: _exchange([s[k] for s in sends], counts) for k in ("x", "ids", "w")}
    host_recv = {k: O.ep_exchange([h[i] for h in host_sends], counts)
                 for k, i in (("x", 2), ("ids", 3), ("w", 4))}
    ys = []
    for r in range(REP_EP):
        R = recv["x"][r].shape[0]
        w13_r = np.stack([w13[e] for e in REP_SLOT_EXPERT[r]])
        w2_r = np.stack([w2[e] for e in REP_SLOT_EXPERT[r]])
        y = torch.zeros(R, REP_H, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(B.ep_expert_compute_workspace_size(cfg[r], R), dtype=torch.uint8,
                         device="cuda")
        B.moe_ep_expert_compute(cfg[r], R, recv["x"][r].contiguous(),
                                recv["ids"][r].contiguous(), recv["w"][r].contiguous(),
                                _dev(w13_r), _dev(w2_r), y, ws)
        assert B.moe_get_status(ws) == (0, 0)
        ref = O.ep_expert_compute(host_recv["x"][r], host_recv["ids"][r], host_recv["w"][r],
                                  w13_r, w2_r, r * REP_SLOTS)
        assert_close(y.float().cpu().numpy(), ref, f"replicas rank {r} expert rows")
        ys.append(y)

    back = [[counts[s][r] for s in range(REP_EP)] for r in range(REP_EP)]
    rets = _exchange(ys, back)
    for r, T in enumerate(tokens):
        out = torch.empty(T, REP_H, dtype=torch.bfloat16, device="cuda")
        cws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        B.moe_ep_combine(cfg[r], T, rets[r].contiguous(), sends[r]["pos"], None, out, cws)
        assert B.moe_get_status(cws) == (0, 0)
        ref = O.moe_forward(xs[r], rw, w13, w2, top_k=REP_K, renormalize=True, router_b=rb)
        assert_close(out.float().cpu().numpy(), ref, f"replicas rank {r} output")


def test_ep_dispatch_flags_bad_ids_and_handles_empty():
    wl = W("ep_bad", T=6, H=128, I=128, E=8, K=2, ep_size=2)
    cfg = cfg_of(wl)
    ids = torch.tensor([[0, 5], [9, 1], [7, -1], [3, 4], [6, 2], [1, 0]], dtype=torch.int32,
                       device="cuda")
    w = torch.rand(6, 2, device="cuda")
    x = torch.randn(6, 128, device="cuda").to(torch.bfloat16)
    n = 12
    counts = torch.empty(2, dtype=torch.int32, device="cuda")
    offsets = torch.empty(3, dtype=torch.int32, device="cuda")
    pos = torch.empty(n, dtype=torch.int32, device="cuda")
    sx = torch.zeros(n, 128, dtype=torch.bfloat16, device="cuda")
    si = torch.empty(n, dtype=torch.int32, device="cuda")
    sw = torch.empty(n, dtype=torch.float32, device="cuda")
    st = torch.empty(n, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.ep_dispatch_workspace_size(cfg, 6), dtype=torch.uint8, device="cuda")
    B.moe_ep_dispatch(cfg, 6, x, ids, w, counts, offsets, pos, sx, si, sw, st, ws)
    rc, flags = B.moe_get_status(ws)
    assert rc == 5 and flags & B.DEV_BAD_EXPERT_ID
    p = pos.cpu().numpy()
    assert p[2] == -1 and p[5] == -1          # ids 9 and -1 are dropped
    # valid ids 0 1 3 2 1 0 -> rank 0, ids 5 7 4 6 -> rank 1
    assert counts.cpu().numpy().tolist() == [6, 4]
    # no tokens: zero counts, nothing else touched
    B.moe_ep_dispatch(cfg, 0, x, ids, w, counts, offsets, pos, sx, si, sw, st, ws)
    torch.cuda.synchronize()
    assert counts.cpu().numpy().tolist() == [0, 0]
    assert offsets.cpu().numpy().tolist() == [0, 0, 0]


def test_ep_expert_compute_full_shard_sampled():
    """One rank's expert compute at the EP-shard shape (H=2048, I=512, E=256,
    ep 4, rank 1): 66,049 received items over the 64 local experts, skewed,
    two experts without items, so segments run to thousands of rows (256-row
    tiles on CTA pairs) with ragged ends, and 40 items whose expert belongs to
    another rank (their rows must come back zero). Each returned row depends
    on its own item only, so sampled rows are checked against the oracle."""
    wl = synth.EP_SHARD
    El, e0, H, I = wl.E_local, wl.ep_rank * wl.E_local, wl.H, wl.I
    R = 66049
    rng = np.random.default_rng(7)
    pop = rng.dirichlet(np.full(El, 0.7))
    pop[[5, 40]] = 0.0
    lid = rng.choice(El, size=R, p=pop / pop.sum()).astype(np.int32)
    ids = lid + e0
    foreign = rng.choice(R, size=40, replace=False)
    ids[foreign] = rng.choice(np.r_[0:e0, e0 + El:wl.E], size=40)
    lid[foreign] = -1
    w = rng.uniform(0.05, 1.0, size=R).astype(np.float32)
    x = synth.draw(3, synth.X, 0, R, H, wl.std(synth.X), True)
    w13b = synth.draw_bf16_bits(0, synth.W13, e0 * 2 * I, El * 2 * I, H,
                                wl.std(synth.W13)).reshape(El, 2 * I, H)
    w2b = synth.draw_bf16_bits(0, synth.W2, e0 * H, El * H, I,
                               wl.std(synth.W2)).reshape(El, H, I)
    cfg = cfg_of(wl)
    y = torch.full((R, H), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(B.ep_expert_compute_workspace_size(cfg, R), dtype=torch.uint8,
                     device="cuda")
    B.moe_ep_expert_compute(cfg, R, _dev(x), torch.from_numpy(ids).cuda(),
                            torch.from_numpy(w).cuda(),
                            torch.from_numpy(w13b.view(np.int16)).view(torch.bfloat16).cuda(),
                            torch.from_numpy(w2b.view(np.int16)).view(torch.bfloat16).cuda(),
                            y, ws)
    assert B.moe_get_status(ws) == (0, 0)
    # every local expert's first and last item, plus an even spread
    rows = set(np.linspace(0, R - 1, 256).astype(np.int64).tolist())
    for e in range(El):
        hit = np.nonzero(lid == e)[0]
        if hit.size:
            rows.update((int(hit[0]), int(hit[-1])))
    rows = np.array(sorted(rows.difference(foreign.tolist())))
    w13h, w2h = synth.BF16Experts(w13b), synth.BF16Experts(w2b)
    ref = O.ep_expert_compute(x[rows], ids[rows], w[rows], w13h, w2h, e0)
    yh = y.float().cpu().numpy()
    assert_close(yh[rows], ref, "EP-shard expert rows")
    assert not yh[foreign].any(), "rows of other ranks' items must be zero"
