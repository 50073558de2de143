"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Every check compares the oracle with something independent of it: a closed
form, a library routine (scipy, numpy.array_split), a brute-force
pure-Python implementation on tiny inputs, an algebraic identity between two
different formulations, or the figures the pages print. At the end,
planted-mistake tests show that these checks catch plausible errors.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import moe_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(1234)


def _layer(T=6, H=12, I=10, E=8, S=0, Is=6, seed=0, bias=False):
    r = np.random.default_rng(seed)
    d = dict(x=r.standard_normal((T, H)),
             router_w=r.standard_normal((E, H)) * 0.7,
             router_b=r.standard_normal(E) if bias else None,
             w13=r.standard_normal((E, 2 * I, H)) / math.sqrt(H),
             w2=r.standard_normal((E, H, I)) / math.sqrt(I),
             shared_w13=r.standard_normal((S, 2 * Is, H)) / math.sqrt(H) if S else None,
             shared_w2=r.standard_normal((S, H, Is)) / math.sqrt(Is) if S else None)
    return d


def _fwd(d, **kw):
    return O.moe_forward(d["x"], d["router_w"], d["w13"], d["w2"],
                         router_b=d["router_b"], shared_w13=d["shared_w13"],
                         shared_w2=d["shared_w2"], **kw)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------
def test_softmax_matches_scipy():
    lg = (RNG.standard_normal((50, 256)) * 3).astype(np.float32)
    p = O.softmax_fp32(lg)
    ref = scipy.special.softmax(lg.astype(np.float64), axis=1)
    np.testing.assert_allclose(p, ref, rtol=2e-6, atol=1e-9)
    assert p.dtype == np.float32


def test_router_logits_are_x_times_wg_transpose():
    # non-square shapes: a transposed operand cannot even be multiplied
    x = RNG.standard_normal((5, 7)).astype(np.float32)
    wg = RNG.standard_normal((3, 7)).astype(np.float32)
    b = RNG.standard_normal(3).astype(np.float32)
    lg = O.router_logits(x, wg, b)
    assert lg.shape == (5, 3)
    for t in range(5):
        for e in range(3):
            ref = math.fsum(float(x[t, h]) * float(wg[e, h]) for h in range(7)) + float(b[e])
            assert abs(float(lg[t, e]) - ref) <= 1e-6 * max(1.0, abs(ref))


def _brute_topk(prow, k, eligible=None):
    """Rank by counting: e is chosen iff fewer than k eligible experts beat it."""
    E = len(prow)
    elig = list(range(E)) if eligible is None else eligible
    def beats(a, b):
        return prow[a] > prow[b] or (prow[a] == prow[b] and a < b)
    ranked = []
    for e in elig:
        better = sum(1 for f in elig if f != e and beats(f, e))
        if better < k:
            ranked.append((better, e))
    return [e for _, e in sorted(ranked)]


def test_topk_plain_brute_force_with_ties():
    # quantised probabilities force many exact ties
    p = (RNG.integers(0, 5, size=(200, 10)) / 8.0).astype(np.float32)
    for k in (1, 3, 10):
        ids = O.topk_plain(p, k)
        for t in range(p.shape[0]):
            assert list(ids[t]) == _brute_topk(list(p[t]), k)


def _brute_grouped(prow, k, n_group, topk_group):
    E = len(prow)
    gs = E // n_group
    score = [max(prow[g * gs:(g + 1) * gs]) for g in range(n_group)]
    def gbeats(a, b):
        return score[a] > score[b] or (score[a] == score[b] and a < b)
    kept = [g for g in range(n_group)
            if sum(1 for h in range(n_group) if h != g and gbeats(h, g)) < topk_group]
    elig = [e for e in range(E) if e // gs in kept]
    return _brute_topk(prow, k, elig)


def _subset_grouped(prow, k, n_group, topk_group):
    """Brute force over all C(n_group, topk_group) subsets of groups.

    The kept subset is the one whose scores, sorted descending with the group
    ids as tie-break, are lexicographically best."""
    E = len(prow)
    gs = E // n_group
    score = [max(prow[g * gs:(g + 1) * gs]) for g in range(n_group)]
    best, best_key = None, None
    for sub in itertools.combinations(range(n_group), topk_group):
        key = sorted(((-score[g], g) for g in sub))
        if best_key is None or key < best_key:
            best, best_key = sub, key
    elig = [e for e in range(E) if e // gs in best]
    return _brute_topk(prow, k, elig)


@pytest.mark.parametrize("E,n_group,topk_group,k", [(8, 4, 2, 3), (12, 3, 1, 2),
                                                   (16, 4, 3, 5), (8, 2, 1, 4)])
def test_grouped_topk_brute_force(E, n_group, topk_group, k):
    p = (RNG.integers(0, 7, size=(150, E)) / 16.0).astype(np.float32)
    ids = O.topk_grouped(p, k, n_group, topk_group)
    for t in range(p.shape[0]):
        assert list(ids[t]) == _brute_grouped(list(p[t]), k, n_group, topk_group)
        assert list(ids[t]) == _subset_grouped(list(p[t]), k, n_group, topk_group)


def test_grouped_topk_reduces_to_plain():
    p = O.softmax_fp32(RNG.standard_normal((100, 32)).astype(np.float32))
    for k in (1, 4, 8):
        plain = O.topk_plain(p, k)
        np.testing.assert_array_equal(O.topk_grouped(p, k, 8, 8), plain)
        np.testing.assert_array_equal(O.topk_grouped(p, k, 1, 1), plain)


def test_route_weights_renormalised_and_raw():
    d = _layer(T=20, E=16)
    ids, w, p = O.route(d["x"], d["router_w"], top_k=4, renormalize=True)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-6)
    ids2, w2, _ = O.route(d["x"], d["router_w"], top_k=4, renormalize=False)
    np.testing.assert_array_equal(ids, ids2)
    ref = scipy.special.softmax(O.router_logits(d["x"], d["router_w"]).astype(np.float64), axis=1)
    np.testing.assert_allclose(w2, np.take_along_axis(ref, ids, 1), rtol=2e-6)
    # descending order
    assert (np.diff(w2, axis=1) <= 0).all()


def _router_for_logits(logits):
    """x = identity rows, router = the logits as its first column: the oracle's
    logits are then exactly the given values."""
    l = np.asarray(logits, np.float64)
    T, E = l.shape
    return np.eye(T, T + 1), np.concatenate([l.T, np.zeros((E, 1))], axis=1)


def test_sigmoid_scores_closed_form():
    l = np.array([[0.0, math.log(3.0), -math.log(3.0), math.log(1 / 9)]], np.float32)
    np.testing.assert_allclose(O.sigmoid_fp32(l), [[0.5, 0.75, 0.25, 0.1]], rtol=1e-6)
    np.testing.assert_allclose(O.sigmoid_fp32(l), scipy.special.expit(l.astype(np.float64)),
                               rtol=1e-6)


def test_route_sigmoid_hand_example():
    # sigmoid scores 0.5, 0.75, 0.25, 0.1: top-2 = experts 1, 0
    x, rw = _router_for_logits([[0.0, math.log(3.0), -math.log(3.0), math.log(1 / 9)]])
    ids, w, sel = O.route(x, rw, top_k=2, renormalize=False, scoring="sigmoid")
    assert list(ids[0]) == [1, 0]
    np.testing.assert_allclose(w[0], [0.75, 0.5], rtol=1e-6)
    _, wr, _ = O.route(x, rw, top_k=2, renormalize=True, scoring="sigmoid")
    np.testing.assert_allclose(wr[0], [0.6, 0.4], rtol=1e-6)


def test_selection_bias_changes_choice_not_weights():
    # scores 0.5, 0.75, 0.25, 0.1; correction +0.6 on expert 2 -> selection
    # scores 0.5, 0.75, 0.85, 0.1: experts 2, 1 are chosen, with their
    # uncorrected scores 0.25, 0.75 as weights
    x, rw = _router_for_logits([[0.0, math.log(3.0), -math.log(3.0), math.log(1 / 9)]])
    b = np.array([0.0, 0.0, 0.6, 0.0])
    ids, w, sel = O.route(x, rw, b, top_k=2, renormalize=False, scoring="sigmoid",
                          bias_mode="select")
    assert list(ids[0]) == [2, 1]
    np.testing.assert_allclose(w[0], [0.25, 0.75], rtol=1e-6)
    np.testing.assert_allclose(sel[0], [0.5, 0.75, 0.85, 0.1], rtol=1e-6)
    _, wr, _ = O.route(x, rw, b, top_k=2, renormalize=True, scoring="sigmoid",
                       bias_mode="select")
    np.testing.assert_allclose(wr[0], [0.25, 0.75], rtol=1e-6)  # already sums to 1
    # the same bias as a logit bias moves the weights as well
    _, wl, _ = O.route(x, rw, b, top_k=2, renormalize=False, scoring="sigmoid",
                       bias_mode="logit")
    assert not np.allclose(wl[0], w[0])


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
def test_zero_selection_bias_is_plain_routing(scoring):
    d = _layer(T=30, E=16, seed=5)
    for kw in (dict(), dict(n_group=4, topk_group=2)):
        ref = O.route(d["x"], d["router_w"], top_k=3, renormalize=True, scoring=scoring, **kw)
        got = O.route(d["x"], d["router_w"], np.zeros(16), top_k=3, renormalize=True,
                      scoring=scoring, bias_mode="select", **kw)
        for a, b in zip(ref, got):
            np.testing.assert_array_equal(a, b)


def test_sigmoid_choice_follows_logit_order():
    d = _layer(T=60, E=24, seed=6)
    lg = O.router_logits(d["x"], d["router_w"])
    ids, w, _ = O.route(d["x"], d["router_w"], top_k=5, renormalize=False, scoring="sigmoid")
    for t in range(60):
        assert list(ids[t]) == _brute_topk(list(lg[t]), 5, range(24))
    np.testing.assert_allclose(w, scipy.special.expit(np.take_along_axis(lg, ids, 1)
                                                      .astype(np.float64)), rtol=1e-6)


def test_grouped_selection_bias_brute_force():
    r = np.random.default_rng(11)
    for _ in range(40):
        l = r.standard_normal((1, 16)).astype(np.float32)
        b = (r.integers(-3, 4, size=16) / 8.0)
        x, rw = _router_for_logits(l)
        ids, w, sel = O.route(x, rw, b, top_k=3, renormalize=False, scoring="sigmoid",
                              bias_mode="select", n_group=4, topk_group=2)
        p = scipy.special.expit(l[0].astype(np.float64))
        s32 = (p.astype(np.float32) + b.astype(np.float32)).astype(np.float32)
        assert list(ids[0]) == _subset_grouped(list(s32), 3, 4, 2)
        np.testing.assert_allclose(w[0], p[ids[0]], rtol=1e-6)


def test_min_gap_detects_near_ties():
    p = np.array([[0.5, 0.3, 0.2 + 5e-6, 0.2 - 5e-6],
                  [0.4, 0.3, 0.2, 0.1]], dtype=np.float64)
    g = O.routing_min_gap(p, 2)
    assert g[1] == pytest.approx(0.1)
    assert g[0] == pytest.approx(0.3 - (0.2 + 5e-6))  # k=2 boundary: 0.3 vs 0.2+5e-6
    g3 = O.routing_min_gap(p, 3)
    assert g3[0] < 2e-5


# ---------------------------------------------------------------------------
# expert MLP
# ---------------------------------------------------------------------------
def test_silu_closed_form():
    z = np.linspace(-30, 30, 601)
    s = O.silu(z)
    np.testing.assert_allclose(s, z * scipy.special.expit(z), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(s - O.silu(-z), z, rtol=1e-12, atol=1e-12)
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(50.0) - 50.0) < 1e-12
    assert abs(O.silu(-50.0)) < 1e-18


def test_gate_up_roles_and_down_layout():
    # H=4, I=2: gate rows saturate silu (silu(30) ~ 30), up rows are distinct
    H, I = 4, 2
    x = np.array([[1.0, 0.0, 0.0, 0.0]])
    w13 = np.zeros((2 * I, H))
    w13[0:I, 0] = 30.0                 # gate rows [0, I)
    w13[I:2 * I, 0] = [1.0, 2.0]       # up rows [I, 2I)
    w2 = np.zeros((H, I))              # [out=H, in=I]
    w2[0, 0], w2[1, 1], w2[3, 0] = 1.0, 1.0, -2.0
    y = O.expert_mlp(x, w13, w2)[0]
    h = np.array([30.0, 60.0]) * (1 - math.exp(-30))  # silu(30)*u, up to e^-30
    np.testing.assert_allclose(y, [h[0], h[1], 0.0, -2 * h[0]], rtol=1e-9)


# ---------------------------------------------------------------------------
# forward: identities between formulations
# ---------------------------------------------------------------------------
CONFIGS = [
    dict(top_k=2, renormalize=True),
    dict(top_k=3, renormalize=False, rsf=2.5),
    dict(top_k=3, renormalize=True, n_group=4, topk_group=2),
    dict(top_k=2, renormalize=False, n_group=2, topk_group=1, rsf=16.0),
]


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("shared", [0, 2])
def test_sum_over_k_equals_page_masked_loop(cfg, shared):
    d = _layer(T=9, E=8, S=shared, bias=True)
    a = _fwd(d, **cfg)
    b = O.moe_forward_masked_loop(d["x"], d["router_w"], d["w13"], d["w2"],
                                  router_b=d["router_b"], shared_w13=d["shared_w13"],
                                  shared_w2=d["shared_w2"], **cfg)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_masked_loop_with_ep_map():
    d = _layer(T=9, E=8)
    for r in range(4):
        em = O.expert_map(8, 4, r)
        loc = {k: v[2 * r:2 * r + 2] for k, v in d.items() if k in ("w13", "w2")}
        a = O.moe_forward(d["x"], d["router_w"], loc["w13"], loc["w2"], top_k=3, emap=em)
        b = O.moe_forward_masked_loop(d["x"], d["router_w"], loc["w13"], loc["w2"],
                                      top_k=3, emap=em)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_full_topk_is_softmax_mixture():
    """top_k = E with renormalise gives sum_e softmax_e * f_e(x)."""
    d = _layer(T=7, E=6)
    out = _fwd(d, top_k=6, renormalize=True)
    lg = d["x"] @ d["router_w"].T
    p = scipy.special.softmax(lg, axis=1)
    ref = sum(p[:, e:e + 1] * O.expert_mlp(d["x"], d["w13"][e], d["w2"][e]) for e in range(6))
    np.testing.assert_allclose(out, ref, rtol=2e-6, atol=1e-7)
    _, w, _ = O.route(d["x"], d["router_w"], top_k=6, renormalize=True)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-6)


@pytest.mark.parametrize("ep", [1, 2, 4, 8])
def test_ep_shard_sum_equals_unsharded(ep):
    d = _layer(T=11, E=8, S=2, bias=True)
    full = _fwd(d, top_k=3, renormalize=True, rsf=1.5)
    acc = np.zeros_like(full)
    El = 8 // ep
    for r in range(ep):
        em = O.expert_map(8, ep, r)
        acc += O.moe_forward(d["x"], d["router_w"], d["w13"][r * El:(r + 1) * El],
                             d["w2"][r * El:(r + 1) * El], top_k=3, renormalize=True,
                             rsf=1.5, router_b=d["router_b"], emap=em,
                             shared_w13=d["shared_w13"] if r == 0 else None,
                             shared_w2=d["shared_w2"] if r == 0 else None)
    np.testing.assert_allclose(acc, full, rtol=1e-12, atol=1e-12)


# A global placement with redundant experts over 2 ranks: logical experts 0-7,
# experts 2 and 5 replicated (expert 2 three times). Each rank holds physical
# slots; a slot carries its logical expert's weights.
_PLACEMENT = [[(0, 0)], [(0, 1)], [(0, 2), (1, 4), (0, 5)], [(0, 3)],
              [(1, 0)], [(1, 1), (0, 4)], [(1, 2)], [(1, 3)]]
_SLOTS = [[0, 1, 2, 3, 5, 2], [4, 5, 6, 7, 2]]   # logical expert of each slot, per rank


def test_replica_maps_partition_items_and_sum_to_unsharded():
    """Redundant experts: every (token, slot) item lands on exactly one replica
    across the ranks, a hot expert's items spread round robin over its
    replicas, and the ranks' partial outputs add up to the unsharded layer
    (the replicas hold the same weights)."""
    d = _layer(T=13, E=8, S=1, bias=True)
    kw = dict(top_k=3, renormalize=True, rsf=1.5)
    full = _fwd(d, **kw)
    kw["router_b"] = d["router_b"]
    maps = O.replica_maps(_PLACEMENT, 2, 3)
    ids, _, _ = O.route(d["x"], d["router_w"], d["router_b"], top_k=3, renormalize=True)
    hits = np.zeros(ids.shape, dtype=np.int64)
    acc = np.zeros_like(full)
    for r in range(2):
        loc = O.local_slots(ids, maps[r])
        hits += loc >= 0
        for t, k in zip(*np.nonzero(loc >= 0)):
            assert _SLOTS[r][loc[t, k]] == ids[t, k]       # the slot holds that expert
        w13 = np.stack([d["w13"][e] for e in _SLOTS[r]])
        w2 = np.stack([d["w2"][e] for e in _SLOTS[r]])
        acc += O.moe_forward(d["x"], d["router_w"], w13, w2, emap=maps[r],
                             shared_w13=d["shared_w13"] if r == 0 else None,
                             shared_w2=d["shared_w2"] if r == 0 else None, **kw)
    np.testing.assert_array_equal(hits, 1)
    np.testing.assert_allclose(acc, full, rtol=1e-12, atol=1e-12)
    # expert 2's items: token t uses replica t mod 3
    for t, k in zip(*np.nonzero(ids == 2)):
        rank, slot = _PLACEMENT[2][t % 3]
        assert O.local_slots(ids, maps[rank])[t, k] == slot


def test_one_replica_map_equals_plain_map_and_bad_rows_are_refused():
    d = _layer(T=9, E=8)
    em = O.expert_map(8, 2, 1)
    rmap = np.full((8, 2), O.NO_REPLICA, dtype=np.int32)
    rmap[:, 0] = em
    ids, _, _ = O.route(d["x"], d["router_w"], None, top_k=2, renormalize=True)
    np.testing.assert_array_equal(O.local_slots(ids, rmap), em[ids])
    a = O.align_permute(ids, em, 4, 16)
    b = O.align_permute(ids, rmap, 4, 16)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
    bad = rmap.copy()
    bad[int(ids[0, 0])] = O.NO_REPLICA            # an expert without replicas
    with pytest.raises(ValueError):
        O.local_slots(ids, bad)
    with pytest.raises(ValueError):
        O.replica_maps([[(0, 0)] * 4], 1, 3)      # more replicas than max_replicas


def test_expert_map_matches_array_split_and_page_example():
    for E, ep in [(8, 2), (256, 4), (160, 8), (64, 8)]:
        for r in range(ep):
            em = O.expert_map(E, ep, r)
            mine = np.nonzero(em >= 0)[0]
            np.testing.assert_array_equal(mine, np.array_split(np.arange(E), ep)[r])
            np.testing.assert_array_equal(em[mine], np.arange(E // ep))
    g = json.load(open(os.path.join(HERE, "golden", "ep_weight_sizing.json")))["local_experts"]
    assert (O.expert_map(g["num_experts"], g["ep_size"], 0) >= 0).sum() == g["num_local_experts"]
    with pytest.raises(ValueError):
        O.expert_map(10, 4, 0)


def test_two_shared_experts_equal_one_merged():
    d = _layer(T=5, S=2, Is=6)
    a = _fwd(d, top_k=2)
    s13, s2 = d["shared_w13"], d["shared_w2"]
    Is = s2.shape[2]
    merged13 = np.concatenate([s13[0][:Is], s13[1][:Is], s13[0][Is:], s13[1][Is:]])[None]
    merged2 = np.concatenate([s2[0], s2[1]], axis=1)[None]
    d2 = dict(d, shared_w13=merged13, shared_w2=merged2)
    b = _fwd(d2, top_k=2)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_rsf_scales_routed_part_only():
    d = _layer(T=5, S=1)
    shared = sum(O.expert_mlp(d["x"], d["shared_w13"][s], d["shared_w2"][s]) for s in range(1))
    one = _fwd(d, top_k=2, rsf=1.0) - shared
    sixteen = _fwd(d, top_k=2, rsf=16.0) - shared
    np.testing.assert_allclose(sixteen, 16.0 * one, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# brute force, pure Python scalar loops, tiny inputs
# ---------------------------------------------------------------------------
def _brute_forward(x, rw, rb, w13, w2, K, renorm, n_group, topk_group, rsf, emap,
                   sw13=None, sw2=None):
    T, H = x.shape
    E = rw.shape[0]
    I = w2.shape[2]

    def mlp(xt, a13, a2, Ii):
        h = []
        for i in range(Ii):
            g = math.fsum(a13[i][c] * xt[c] for c in range(H))
            u = math.fsum(a13[Ii + i][c] * xt[c] for c in range(H))
            h.append(g / (1.0 + math.exp(-g)) * u)
        return [math.fsum(a2[o][i] * h[i] for i in range(Ii)) for o in range(H)]

    out = []
    for t in range(T):
        xt = [float(v) for v in x[t]]
        lg = [math.fsum(xt[c] * float(rw[e][c]) for c in range(H)) + (float(rb[e]) if rb is not None else 0.0)
              for e in range(E)]
        mx = max(lg)
        ex = [math.exp(v - mx) for v in lg]
        s = math.fsum(ex)
        p = [v / s for v in ex]
        chosen = _brute_grouped(p, K, n_group, topk_group) if n_group else _brute_topk(p, K)
        w = [p[e] for e in chosen]
        if renorm:
            sw = math.fsum(w)
            w = [v / sw for v in w]
        acc = [0.0] * H
        for e, we in zip(chosen, w):
            le = int(emap[e])
            if le < 0:
                continue
            y = mlp(xt, w13[le], w2[le], I)
            acc = [a + we * yv for a, yv in zip(acc, y)]
        acc = [rsf * a for a in acc]
        if sw13 is not None:
            for s_ in range(sw13.shape[0]):
                y = mlp(xt, sw13[s_], sw2[s_], sw2.shape[2])
                acc = [a + yv for a, yv in zip(acc, y)]
        out.append(acc)
    return np.array(out)


BRUTE = [
    dict(E=8, K=2, renorm=True, n_group=0, topk_group=0, rsf=1.0, ep=(1, 0), S=0),
    dict(E=8, K=3, renorm=False, n_group=4, topk_group=2, rsf=16.0, ep=(1, 0), S=2),
    dict(E=8, K=2, renorm=True, n_group=0, topk_group=0, rsf=1.0, ep=(4, 1), S=0),
    dict(E=6, K=6, renorm=True, n_group=0, topk_group=0, rsf=1.0, ep=(2, 1), S=1),
]


def _brute_case(c, seed=3):
    d = _layer(T=4, H=10, I=7, E=c["E"], S=c["S"], Is=5, seed=seed, bias=True)
    ep, r = c["ep"]
    El = c["E"] // ep
    em = O.expert_map(c["E"], ep, r)
    w13, w2 = d["w13"][r * El:(r + 1) * El], d["w2"][r * El:(r + 1) * El]
    kw = dict(top_k=c["K"], renormalize=c["renorm"], n_group=c["n_group"],
              topk_group=c["topk_group"], rsf=c["rsf"], router_b=d["router_b"],
              shared_w13=d["shared_w13"], shared_w2=d["shared_w2"], emap=em)
    ref = _brute_forward(d["x"], d["router_w"], d["router_b"], w13, w2, c["K"], c["renorm"],
                         c["n_group"], c["topk_group"], c["rsf"], em,
                         d["shared_w13"], d["shared_w2"])
    return d, w13, w2, kw, ref


@pytest.mark.parametrize("c", BRUTE)
def test_forward_brute_force_tiny(c):
    d, w13, w2, kw, ref = _brute_case(c)
    out = O.moe_forward(d["x"], d["router_w"], w13, w2, **kw)
    # the oracle's softmax is fp32 (the page's precision); brute force is fp64
    np.testing.assert_allclose(out, ref, rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------------------
# alignment / permutation
# ---------------------------------------------------------------------------
def _brute_align(ids, emap, El, block):
    T, K = ids.shape
    items = [(int(emap[ids[t, k]]), t * K + k) for t in range(T) for k in range(K)]
    items = sorted(i for i in items if i[0] >= 0)
    counts = [sum(1 for e, _ in items if e == le) for le in range(El)]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + ((c + block - 1) // block) * block)
    rows = {}
    for le in range(El):
        mine = [it for e, it in items if e == le]
        for j, it in enumerate(mine):
            rows[offsets[le] + j] = it
    return counts, offsets, rows


@pytest.mark.parametrize("T,K,E,ep,r,block", [(13, 2, 8, 1, 0, 16), (40, 4, 16, 4, 2, 8),
                                             (7, 3, 6, 2, 1, 1), (1, 8, 256, 1, 0, 16),
                                             (0, 2, 8, 1, 0, 16), (64, 8, 256, 4, 1, 128)])
def test_align_permute_brute_force(T, K, E, ep, r, block):
    ids = np.array([RNG.permutation(E)[:K] for _ in range(T)], dtype=np.int32).reshape(T, K)
    El = E // ep
    em = O.expert_map(E, ep, r)
    counts, offsets, sorted_ids, inv_pos = O.align_permute(ids, em, El, block)
    bc, bo, rows = _brute_align(ids, em, El, block)
    np.testing.assert_array_equal(counts, bc)
    np.testing.assert_array_equal(offsets, bo)
    cap = O.align_cap(T, K, El, block)
    assert len(sorted_ids) == cap and offsets[-1] <= cap
    for row in range(cap):
        assert sorted_ids[row] == rows.get(row, T * K)
    for it in range(T * K):
        if inv_pos[it] >= 0:
            assert sorted_ids[inv_pos[it]] == it
        else:
            assert em[ids.reshape(-1)[it]] < 0
    assert (np.asarray(offsets) % block == 0).all()
    # per-rank counts sum to T*K over all ranks (every item lands on one rank)
    if ep > 1:
        tot = sum(O.align_permute(ids, O.expert_map(E, ep, q), El, block)[0].sum()
                  for q in range(ep))
        assert tot == T * K


def test_grouped_mlp_and_combine_recompose_forward():
    d = _layer(T=10, E=8, S=1)
    ids, w, _ = O.route(d["x"], d["router_w"], top_k=3, renormalize=False)
    em = O.expert_map(8, 2, 1)
    w13, w2 = d["w13"][4:], d["w2"][4:]
    counts, offsets, sorted_ids, inv_pos = O.align_permute(ids, em, 4, 4)
    ys = O.grouped_mlp(d["x"], sorted_ids, offsets, w13, w2, 3)
    y = np.full((len(sorted_ids), d["x"].shape[1]), np.nan)
    for row, v in ys.items():
        y[row] = v
    shared = O.expert_mlp(d["x"], d["shared_w13"][0], d["shared_w2"][0])
    out = O.combine(y, inv_pos, w, rsf=4.0, shared_out=shared)
    ref = O.moe_forward(d["x"], d["router_w"], w13, w2, top_k=3, renormalize=False,
                        rsf=4.0, emap=em, shared_w13=d["shared_w13"], shared_w2=d["shared_w2"])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# the pages' printed figures
# ---------------------------------------------------------------------------
def _ep_pipeline(rank_x, d, ep, top_k, rsf=1.0, routing_kw=None, combine=None):
    """Every rank routes its own tokens globally, dispatches, exchanges, runs
    its expert shard, returns and combines (host-simulated all-to-alls)."""
    E = d["router_w"].shape[0]
    El = E // ep
    kw = dict(top_k=top_k, renormalize=True, **(routing_kw or {}))
    sends = []
    for x in rank_x:
        ids, w, _ = O.route(x, d["router_w"], d["router_b"], **kw)
        sends.append(O.ep_dispatch(x, ids, w, E, ep))
    counts = [s[0] for s in sends]
    recv_x = O.ep_exchange([s[2] for s in sends], counts)
    recv_ids = O.ep_exchange([s[3] for s in sends], counts)
    recv_w = O.ep_exchange([s[4] for s in sends], counts)
    outs = [O.ep_expert_compute(recv_x[r], recv_ids[r], recv_w[r],
                                d["w13"][r * El:(r + 1) * El], d["w2"][r * El:(r + 1) * El],
                                r * El) for r in range(ep)]
    back_counts = [[counts[s][r] for s in range(ep)] for r in range(ep)]
    ret = O.ep_exchange(outs, back_counts)
    comb = combine or O.ep_combine
    res = []
    for r, x in enumerate(rank_x):
        sh = None
        if d["shared_w13"] is not None:
            sh = sum(O.expert_mlp(x, d["shared_w13"][s], d["shared_w2"][s])
                     for s in range(d["shared_w13"].shape[0]))
        res.append(comb(ret[r], sends[r][1], top_k, rsf, sh))
    return res


@pytest.mark.parametrize("ep", [2, 4])
def test_ep_dispatch_pipeline_equals_unsharded(ep):
    d = _layer(T=1, H=12, I=10, E=8, S=1, seed=21, bias=True)
    r = np.random.default_rng(22)
    rank_x = [r.standard_normal((n, 12)) for n in (7, 0, 5, 9)[:ep]]
    for kw in (dict(), dict(n_group=4, topk_group=2)):
        got = _ep_pipeline(rank_x, d, ep, 3, rsf=1.5, routing_kw=kw)
        for x, g in zip(rank_x, got):
            ref = _fwd(dict(d, x=x), top_k=3, rsf=1.5, **kw)
            np.testing.assert_allclose(g, ref, rtol=1e-12, atol=1e-12)


def test_ep_dispatch_brute_force():
    r = np.random.default_rng(23)
    T, K, E, ep = 13, 3, 12, 4
    ids = np.stack([r.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    w = r.random((T, K)).astype(np.float32)
    x = r.standard_normal((T, 5))
    counts, pos, sx, sid, sw, stok = O.ep_dispatch(x, ids, w, E, ep)
    # brute force: walk items in order, append each to its destination's list
    lists = [[] for _ in range(ep)]
    for t in range(T):
        for k in range(K):
            lists[ids[t, k] // (E // ep)].append((t, k))
    order = [it for l in lists for it in l]
    assert list(counts) == [len(l) for l in lists]
    for row, (t, k) in enumerate(order):
        assert pos[t * K + k] == row and sid[row] == ids[t, k] and stok[row] == t
        assert sw[row] == w[t, k]
        np.testing.assert_array_equal(sx[row], x[t])


def test_ep_dispatch_with_replicas_brute_force():
    """Redundant experts in the token-dispatch form: each item goes to the rank
    of replica t mod n_e of its expert (the local_slots reading), its physical
    id travels in send_ids, and the items a rank receives are exactly those its
    own replica map keeps, at the same slots."""
    r = np.random.default_rng(31)
    T, K, E, ep, n_local = 17, 3, 8, 2, 6
    ids = np.stack([r.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    for t in range(0, T, 2):                  # expert 2 (three replicas) is hot
        if 2 not in ids[t]:
            ids[t, 0] = 2
    w = r.random((T, K)).astype(np.float32)
    x = r.standard_normal((T, 5))
    pmap = O.physical_map(_PLACEMENT, ep, n_local, 3)
    counts, pos, sx, sid, sw, stok = O.ep_dispatch(x, ids, w, E, ep, pmap, n_local)
    lists = [[] for _ in range(ep)]
    for t in range(T):
        for k in range(K):
            reps = _PLACEMENT[ids[t, k]]
            rank, slot = reps[t % len(reps)]
            lists[rank].append((t, k, rank * n_local + slot))
    order = [it for l in lists for it in l]
    assert list(counts) == [len(l) for l in lists]
    for row, (t, k, phys) in enumerate(order):
        assert pos[t * K + k] == row and sid[row] == phys and stok[row] == t
        assert sw[row] == w[t, k]
        np.testing.assert_array_equal(sx[row], x[t])
    maps = O.replica_maps(_PLACEMENT, ep, 3)
    offs = np.concatenate([[0], np.cumsum(counts)])
    item_of_row = np.empty(T * K, dtype=np.int64)
    item_of_row[pos] = np.arange(T * K)
    for rank in range(ep):
        loc = O.local_slots(ids, maps[rank])
        mine = sorted((int(t), int(k)) for t, k in zip(*np.nonzero(loc >= 0)))
        got = [divmod(int(item_of_row[q]), K) for q in range(offs[rank], offs[rank + 1])]
        assert sorted(got) == mine
        for q, (t, k) in zip(range(offs[rank], offs[rank + 1]), got):
            assert sid[q] - rank * n_local == loc[t, k]
    with pytest.raises(ValueError):
        O.physical_map([[(0, 9)]], 1, 4, 1)     # a slot past the rank's slots


def test_ep_dispatch_pipeline_with_replicas_equals_unsharded():
    """All ranks route, dispatch to the replicas, exchange, run their physical
    slots (each holding its logical expert's weights), return and combine: the
    result equals the unsharded layer."""
    d = _layer(T=1, H=12, I=10, E=8, S=1, seed=32, bias=True)
    r = np.random.default_rng(33)
    ep, n_local, K = 2, 6, 3
    pmap = O.physical_map(_PLACEMENT, ep, n_local, 3)
    slot_expert = [[0, 1, 2, 3, 5, 2], [4, 5, 6, 7, 2, 0]]   # rank 1 slot 5 unused
    rank_x = [r.standard_normal((n, 12)) for n in (9, 6)]
    sends = []
    for x in rank_x:
        ids, w, _ = O.route(x, d["router_w"], d["router_b"], top_k=K, renormalize=True)
        sends.append(O.ep_dispatch(x, ids, w, 8, ep, pmap, n_local))
    counts = [s[0] for s in sends]
    recv = [O.ep_exchange([s[i] for s in sends], counts) for i in (2, 3, 4)]
    outs = []
    for rank in range(ep):
        w13 = np.stack([d["w13"][e] for e in slot_expert[rank]])
        w2 = np.stack([d["w2"][e] for e in slot_expert[rank]])
        outs.append(O.ep_expert_compute(recv[0][rank], recv[1][rank], recv[2][rank], w13, w2,
                                        rank * n_local))
    back = [[counts[s][rank] for s in range(ep)] for rank in range(ep)]
    ret = O.ep_exchange(outs, back)
    for rank, x in enumerate(rank_x):
        sh = O.expert_mlp(x, d["shared_w13"][0], d["shared_w2"][0])
        got = O.ep_combine(ret[rank], sends[rank][1], K, 1.5, sh)
        ref = _fwd(dict(d, x=x), top_k=K, rsf=1.5)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_planted_ep_mistakes_are_caught():
    d = _layer(T=1, H=12, I=10, E=8, S=0, seed=24)
    r = np.random.default_rng(25)
    rank_x = [r.standard_normal((6, 12)) for _ in range(2)]
    ref = [_fwd(dict(d, x=x), top_k=2) for x in rank_x]

    def combine_reweighted(ret, pos, k, rsf=1.0, sh=None):
        return 2.0 * O.ep_combine(ret, pos, k, rsf, sh)  # weights applied twice (w ~ 1/2)
    bad = _ep_pipeline(rank_x, d, 2, 2, combine=combine_reweighted)
    assert not all(np.allclose(b, f) for b, f in zip(bad, ref))
    good = _ep_pipeline(rank_x, d, 2, 2)
    assert all(np.allclose(g, f) for g, f in zip(good, ref))


def test_weight_sizing_formula_matches_page():
    g = json.load(open(os.path.join(HERE, "golden", "ep_weight_sizing.json")))
    for c in g["cases"]:
        b = O.weight_bytes_per_card(c["n_experts"], c["intermediate"], c["hidden"],
                                    c["n_layers"], c["elem_bytes"])
        assert b / 2 ** 30 == pytest.approx(c["formula_gib"], abs=1e-9)
    tp2 = g["cases"][0]
    assert tp2["printed_gib"] == tp2["formula_gib"]


# ---------------------------------------------------------------------------
# planted mistakes: each must make an independent check above fail
# ---------------------------------------------------------------------------
def _mutants():
    orig_mlp, orig_route, orig_topk = O.expert_mlp, O.route, O.topk_plain

    def mlp_swapped(x_rows, w13_e, w2_e):
        I = w2_e.shape[1]
        return orig_mlp(x_rows, np.concatenate([w13_e[I:], w13_e[:I]]), w2_e)

    def mlp_sigmoid(x_rows, w13_e, w2_e):
        xr = np.asarray(x_rows, np.float64)
        I = w2_e.shape[1]
        g, u = xr @ w13_e[:I].T, xr @ w13_e[I:].T
        return (scipy.special.expit(g) * u) @ w2_e.T

    def route_no_renorm(*a, **kw):
        kw["renormalize"] = False
        return orig_route(*a, **kw)

    def topk_ties_high(p, k):
        E = p.shape[1]
        return (E - 1 - orig_topk(p[:, ::-1], k)).astype(np.int32)

    def topk_ascending(p, k):
        return orig_topk(p, k)[:, ::-1].copy()

    orig_sig = O.sigmoid_fp32

    def sigmoid_as_tanh(l):
        return np.tanh(np.asarray(l, np.float32)).astype(np.float32)

    def route_weights_corrected(*a, **kw):
        ids, w, sel = orig_route(*a, **kw)
        ws = np.take_along_axis(sel, ids, axis=1).astype(np.float32)
        if kw.get("renormalize"):
            ws = (ws / ws.sum(axis=1, keepdims=True)).astype(np.float32)
        return ids, ws, sel

    return {"expert_mlp": [mlp_swapped, mlp_sigmoid],
            "route": [route_no_renorm, route_weights_corrected],
            "topk_plain": [topk_ties_high, topk_ascending], "sigmoid_fp32": [sigmoid_as_tanh]}


def _brute_checks_pass():
    try:
        for c in BRUTE:
            test_forward_brute_force_tiny(c)
        test_topk_plain_brute_force_with_ties()
        test_gate_up_roles_and_down_layout()
        test_route_weights_renormalised_and_raw()
        test_sigmoid_scores_closed_form()
        test_route_sigmoid_hand_example()
        test_selection_bias_changes_choice_not_weights()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("name,idx", [("expert_mlp", 0), ("expert_mlp", 1), ("route", 0),
                                      ("route", 1), ("topk_plain", 0), ("topk_plain", 1),
                                      ("sigmoid_fp32", 0)])
def test_planted_mistakes_are_caught(monkeypatch, name, idx):
    assert _brute_checks_pass()
    mutant = _mutants()[name][idx]
    monkeypatch.setattr(O, name, mutant)
    assert not _brute_checks_pass(), f"planted mistake in {name} went unnoticed"


def test_planted_combine_and_align_mistakes_are_caught(monkeypatch):
    # rsf applied to the shared output too
    d = _layer(T=5, S=1)
    good = _fwd(d, top_k=2, rsf=3.0)
    orig_mlp = O.expert_mlp
    shared = orig_mlp(d["x"], d["shared_w13"][0], d["shared_w2"][0])
    wrong = 3.0 * (good - shared) + 3.0 * shared
    assert not np.allclose(wrong, good)
    # unstable (descending) order inside a segment is caught by brute force
    ids = np.stack([RNG.permutation(8)[:2] for _ in range(12)]).astype(np.int32)
    em = O.expert_map(8, 1, 0)
    c, o, s, _ = O.align_permute(ids, em, 8, 4)
    bc, bo, rows = _brute_align(ids, em, 8, 4)
    s_bad = s.copy()
    for e in range(8):
        seg = s_bad[o[e]:o[e] + c[e]]
        s_bad[o[e]:o[e] + c[e]] = seg[::-1]
    mism = any(s_bad[r] != v for r, v in rows.items())
    assert mism or all(cc <= 1 for cc in c)
