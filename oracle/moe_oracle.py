"""CPU oracle of the fused MoE layer forward.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module. The CUDA library
never calls it. It shares no code with the CUDA path.

Plain, slow and meant to be read against the source pages. Every function
names the passage it follows. Arithmetic is fp64 except where a page fixes the
precision: the routing softmax is fp32, as in
``F.softmax(router_logits, dim=1, dtype=torch.float)`` (SGLang issue "Expert
parallelism support", MixtralMoE.forward). Router logits are one fp64 dot
product per (token, expert), rounded once to fp32.

Pins (checked by ``tests/test_oracle_pins.py``):
  * routing, top-k, renormalise: pinned by the full-softmax closed form
    (top_k = E), brute-force top-k on tiny inputs, and scipy's softmax;
  * sigmoid scoring and the selection-only score correction: pinned by
    hand-computed examples, by the monotonicity of the sigmoid and by the
    zero-correction identity;
  * grouped top-k: pinned by its reductions to plain top-k and by brute force
    over all group subsets;
  * expert MLP: pinned by the SiLU closed form and the gate/up role test;
  * forward: pinned by the page's dense per-expert masked loop, the EP
    shard-sum identity, shared-expert merging and rsf linearity;
  * align/permute: pinned by a brute-force stable sort and counting;
  * EP dispatch, expert compute, exchange and combine: pinned by the
    all-ranks pipeline equalling the unsharded forward, and by a brute-force
    stable partition by destination rank;
  * redundant experts (replica maps): pinned by the all-ranks sum equalling
    the unsharded forward, by the one-replica map equalling the plain map,
    and by every item landing on exactly one replica.
  The output values themselves have no numeric worked example on the pages,
  so they are pinned only by these identities.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# expert partition (expert parallelism)
# ---------------------------------------------------------------------------
def expert_map(num_experts: int, ep_size: int, ep_rank: int) -> np.ndarray:
    """Global-to-local expert id map of one EP rank, -1 for non-local experts.

    Rank r owns the contiguous range [r*E/ep, (r+1)*E/ep), and local id =
    global id - r*E/ep (ep_fused_moe_patch.py, ``_ep_init``: start_expert_id =
    ep_rank * num_experts_per_rank, with num_experts % ep_size asserted;
    ``_ep_weight_loader``: local_expert_id = expert_id - start; vllm-omni
    "Expert Parallel", Step 4 filters the same range).
    """
    if num_experts % ep_size != 0:
        raise ValueError("num_experts must be divisible by ep_size")
    if not 0 <= ep_rank < ep_size:
        raise ValueError("ep_rank out of range")
    n_local = num_experts // ep_size
    start = ep_rank * n_local
    m = np.full(num_experts, -1, dtype=np.int32)
    m[start:start + n_local] = np.arange(n_local, dtype=np.int32)
    return m


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------
def router_logits(x, router_w, router_b=None) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * Wg[e, h] (+ b[e]), as fp32.

    The gate is a bias-free replicated linear over all global experts
    (MixtralMoE ``self.gate = ReplicatedLinear(hidden, num_experts,
    bias=False)``; vllm-omni "Expert Parallel", Step 2). The optional per-expert
    bias ``b`` is this library's logit-skew input, added before the softmax.
    """
    lg = np.asarray(x, np.float64) @ np.asarray(router_w, np.float64).T
    if router_b is not None:
        lg = lg + np.asarray(router_b, np.float64)[None, :]
    return lg.astype(np.float32)


def softmax_fp32(logits32: np.ndarray) -> np.ndarray:
    """Softmax over experts in fp32 (MixtralMoE.forward, ``dtype=torch.float``)."""
    l = np.asarray(logits32, np.float32)
    m = l.max(axis=1, keepdims=True)
    e = np.exp(l - m)
    return (e / e.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)


def sigmoid_fp32(logits32: np.ndarray) -> np.ndarray:
    """Per-expert sigmoid scores in fp32: 1 / (1 + exp(-l)).

    ``scoring_func`` is named among the FusedMoE routing arguments the pages
    list but not defined there. The reading taken: the non-softmax scoring is
    an elementwise logistic of each logit, in the same fp32 as the softmax.
    """
    l = np.asarray(logits32, np.float32)
    with np.errstate(over="ignore"):
        return (np.float32(1.0) / (np.float32(1.0) + np.exp(-l))).astype(np.float32)


def scores_fp32(logits32: np.ndarray, scoring: str = "softmax") -> np.ndarray:
    """Routing scores p: fp32 softmax over experts, or per-expert sigmoid."""
    if scoring == "softmax":
        return softmax_fp32(logits32)
    if scoring == "sigmoid":
        return sigmoid_fp32(logits32)
    raise ValueError(f"unknown scoring {scoring!r}")


def topk_plain(p: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest p per row, by descending p, ties to the lower id.

    ``torch.topk(routing_weights, top_k, dim=-1)`` (MixtralMoE.forward). A
    stable sort of -p puts equal values in ascending id order.
    """
    order = np.argsort(-p, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def topk_grouped(p: np.ndarray, k: int, n_group: int, topk_group: int) -> np.ndarray:
    """Group-limited top-k (``use_grouped_topk``, ``num_expert_group``, ``topk_group``).

    The pages only name the arguments (vLLM ``MoEMixin.recursive_replace``
    reads ``n_group`` / ``topk_group``; ``ep_fused_moe_patch.py`` passes them to
    ``select_experts``). Reading taken: the E experts form n_group contiguous
    groups of E/n_group. A group scores the max p of its members. The
    topk_group best groups are kept, ties going to the lower group id. Top-k
    then runs over the members of the kept groups only.
    """
    T, E = p.shape
    gs = E // n_group
    gscore = p.reshape(T, n_group, gs).max(axis=2)
    keep_g = np.argsort(-gscore, axis=1, kind="stable")[:, :topk_group]
    keep = np.zeros((T, n_group), dtype=bool)
    keep[np.arange(T)[:, None], keep_g] = True
    masked = np.where(np.repeat(keep, gs, axis=1), p, -np.inf).astype(np.float32)
    return topk_plain(masked, k)


def route(x, router_w, router_b=None, *, top_k, renormalize,
          n_group=0, topk_group=0, scoring="softmax", bias_mode="logit"):
    """(topk_ids [T,K] int32 global ids, topk_w [T,K] fp32, sel [T,E] fp32).

    MixtralMoE.forward: softmax in fp32, topk, then ``routing_weights /=
    routing_weights.sum(dim=-1, keepdim=True)`` when renormalising
    (``renormalize = norm_topk_prob`` in ``MoEMixin.recursive_replace``).
    The weights are the unmasked scores of the chosen experts. Routing is
    global: every rank selects among all experts (ep_fused_moe_patch.py,
    ``_ep_forward`` step 1).

    ``router_b`` has one of two roles (``bias_mode``). "logit": this library's
    skew input, added to the logits before scoring. "select": the per-expert
    score correction that the pages name as ``e_score_correction_bias``
    without defining it. Reading taken: it is added to the scores for choosing
    the groups and the top-k only, and the weights stay the uncorrected
    scores. ``sel`` are the scores the choice was taken on (= p without a
    selection bias).
    """
    if bias_mode not in ("logit", "select"):
        raise ValueError(f"unknown bias_mode {bias_mode!r}")
    logit_b = router_b if bias_mode == "logit" else None
    p = scores_fp32(router_logits(x, router_w, logit_b), scoring)
    sel = p
    if bias_mode == "select" and router_b is not None:
        sel = (p + np.asarray(router_b, np.float32)[None, :]).astype(np.float32)
    if n_group > 0:
        ids = topk_grouped(sel, top_k, n_group, topk_group)
    else:
        ids = topk_plain(sel, top_k)
    w = np.take_along_axis(p, ids, axis=1).astype(np.float32)
    if renormalize:
        w = (w / w.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    return ids, w, sel


def routing_min_gap(p: np.ndarray, top_k: int, n_group: int = 0,
                    topk_group: int = 0) -> np.ndarray:
    """Smallest decision gap per token (for generating tie-free inputs).

    It covers every gap that orders the chosen ids: adjacent ranks among the
    top-k and the k-th vs (k+1)-th. For the grouped variant it also covers the
    group scores up to topk_group and the k-th vs (k+1)-th among kept experts.
    """
    T, E = p.shape
    gaps = []
    if n_group > 0:
        gs = E // n_group
        gscore = np.sort(p.reshape(T, n_group, gs).max(axis=2), axis=1)[:, ::-1]
        upto = min(topk_group, n_group - 1)
        if upto > 0:
            gaps.append(gscore[:, :upto] - gscore[:, 1:upto + 1])
        keep_g = np.argsort(-p.reshape(T, n_group, gs).max(axis=2), axis=1,
                            kind="stable")[:, :topk_group]
        keep = np.zeros((T, n_group), dtype=bool)
        keep[np.arange(T)[:, None], keep_g] = True
        vals = np.where(np.repeat(keep, gs, axis=1), p, -np.inf)
    else:
        vals = p
    s = np.sort(vals, axis=1)[:, ::-1]
    upto = min(top_k, int(np.isfinite(s).sum(axis=1).min()) - 1)
    if upto > 0:
        gaps.append(s[:, :upto] - s[:, 1:upto + 1])
    if not gaps:
        return np.full(T, np.inf)
    return np.concatenate(gaps, axis=1).min(axis=1)


# ---------------------------------------------------------------------------
# expert MLP
# ---------------------------------------------------------------------------
def silu(z):
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z)) (``activation = "silu"``)."""
    z = np.asarray(z, np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_mlp(x_rows, w13_e, w2_e) -> np.ndarray:
    """SiLU-gated expert MLP on rows of x, in fp64.

    f(x) = W2 (silu(W_gate x) * (W_up x)). The stacked ``gate_up_proj`` has
    shape (E, 2*I, H) (vLLM ``MoEMixin.recursive_replace``, packed experts).
    Gate takes rows [0, I) and up takes rows [I, 2I). ``down_proj`` is stored
    [H, I], i.e. [out, in] like gate_up_proj.
    """
    xr = np.asarray(x_rows, np.float64)
    I = w2_e.shape[1]
    g = xr @ np.asarray(w13_e[:I], np.float64).T
    u = xr @ np.asarray(w13_e[I:], np.float64).T
    h = silu(g) * u
    return h @ np.asarray(w2_e, np.float64).T


# ---------------------------------------------------------------------------
# redundant experts: a logical expert with several physical replicas
# ---------------------------------------------------------------------------
REPLICA_ON_OTHER_RANK = -1
NO_REPLICA = -2


def local_slots(ids, emap):
    """Local physical slot of each (token, slot) item, -1 = not on this rank.

    ``emap`` is either the plain map [E] (global id -> local slot or -1,
    ep_fused_moe_patch.py ``_ep_init``) or a replica map [E, R] for redundant
    experts: row e lists the physical replicas of logical expert e in a fixed
    global order, each entry the local slot of a replica on this rank or -1
    for one on another rank, padded with -2. Reading taken, since the pages
    name redundant experts (``num_redundant_experts``) but give no placement
    policy: item (t, k) goes to replica t mod n_e of its expert, with n_e the
    number of replicas, so a hot expert's tokens are spread round robin and
    every item lands on exactly one replica across the ranks. An expert
    without replicas is an error.
    """
    ids = np.asarray(ids)
    emap = np.asarray(emap)
    if emap.ndim == 1:
        return emap[ids]
    T = ids.shape[0]
    loc = np.empty_like(ids, dtype=np.int32)
    for t in range(T):
        for k in range(ids.shape[1]):
            row = emap[ids[t, k]]
            n = int(np.sum(row != NO_REPLICA))
            if n == 0 or np.any(row[:n] == NO_REPLICA):
                raise ValueError("a replica list must be a non-empty prefix of its row")
            loc[t, k] = row[t % n]
    return loc


def replica_maps(placement, ep_size: int, max_replicas: int):
    """Per-rank replica maps [E, R] from a global placement.

    ``placement[e]`` lists (rank, local slot) of each replica of logical
    expert e, in the global replica order. Rank r's map holds the local slot
    for its own replicas and -1 for the others, padded with -2.
    """
    E = len(placement)
    maps = np.full((ep_size, E, max_replicas), NO_REPLICA, dtype=np.int32)
    for e, reps in enumerate(placement):
        if not 1 <= len(reps) <= max_replicas:
            raise ValueError("each expert needs 1..max_replicas replicas")
        for j, (rank, slot) in enumerate(reps):
            maps[:, e, j] = REPLICA_ON_OTHER_RANK
            maps[rank, e, j] = slot
    return maps


def physical_map(placement, ep_size: int, n_local: int, max_replicas: int):
    """Global replica map [E, R] of physical expert ids from a placement.

    ``placement[e]`` lists (rank, local slot) of each replica of logical
    expert e in the global replica order, as for ``replica_maps``. A rank that
    sends tokens to the expert-holding ranks (the EP patch's ``_ep_forward``)
    must know where every replica lives, so this map names each replica by its
    physical id rank * n_local + slot (n_local weight slots per rank), padded
    with -2. It is the placement the per-rank replica maps are cut from.
    """
    E = len(placement)
    pmap = np.full((E, max_replicas), NO_REPLICA, dtype=np.int32)
    for e, reps in enumerate(placement):
        if not 1 <= len(reps) <= max_replicas:
            raise ValueError("each expert needs 1..max_replicas replicas")
        for j, (rank, slot) in enumerate(reps):
            if not (0 <= rank < ep_size and 0 <= slot < n_local):
                raise ValueError("replica outside the physical slots")
            pmap[e, j] = rank * n_local + slot
    return pmap


def physical_ids(ids, pmap):
    """Physical expert id of each (token, slot) item under a global replica
    map: item (t, k) of logical expert e goes to replica t mod n_e of e's n_e
    replicas, the reading ``local_slots`` takes for redundant experts."""
    ids = np.asarray(ids)
    pmap = np.asarray(pmap)
    phys = np.empty_like(ids, dtype=np.int32)
    for t in range(ids.shape[0]):
        for k in range(ids.shape[1]):
            row = pmap[ids[t, k]]
            n = int(np.sum(row != NO_REPLICA))
            if n == 0 or np.any(row[:n] == NO_REPLICA):
                raise ValueError("a replica list must be a non-empty prefix of its row")
            phys[t, k] = row[t % n]
    return phys


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------
def moe_forward(x, router_w, w13, w2, *, top_k, renormalize=True, n_group=0,
                topk_group=0, rsf=1.0, router_b=None, shared_w13=None,
                shared_w2=None, emap=None, tokens=None, routing=None,
                scoring="softmax", bias_mode="logit"):
    """Output rows of the MoE layer for ``tokens`` (default: all), fp64.

    out[t] = rsf * sum_{k : emap[id_tk] >= 0} w_tk * f_{emap[id_tk]}(x_t)
             + sum_s shared_s(x_t)

    This is MixtralMoE.forward's per-expert accumulation written as a sum over
    each token's k slots. ``w13``/``w2`` hold the local experts only, and
    ``emap`` maps global ids to them (ep_fused_moe_patch.py: route globally,
    compute local experts only). ``rsf`` scales the routed sum
    (``routed_scaling_factor``, ``MoEMixin.recursive_replace``). Shared experts
    add unweighted (vllm-omni "Expert Parallel", Step 5).
    """
    x = np.asarray(x)
    T = x.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    if routing is None:
        ids, w, _ = route(x[tok], router_w, router_b, top_k=top_k,
                          renormalize=renormalize, n_group=n_group,
                          topk_group=topk_group, scoring=scoring, bias_mode=bias_mode)
    else:
        ids, w = routing[0][tok], routing[1][tok]
    E_l = w13.shape[0]
    if emap is None:
        emap = np.arange(E_l, dtype=np.int32)
    if np.asarray(emap).ndim == 1:
        loc = np.asarray(emap)[ids]                   # [n, K], -1 = not local
    else:  # replica map: the token index picks the replica
        full = np.zeros((T, ids.shape[1]), dtype=ids.dtype)
        full[tok] = ids
        loc = local_slots(full, emap)[tok]
    f = np.zeros(ids.shape + (x.shape[1],), dtype=np.float64)
    for e in range(E_l):
        rows, slots = np.nonzero(loc == e)
        if rows.size:
            f[rows, slots] = expert_mlp(x[tok[rows]], w13[e], w2[e])
    routed = np.zeros((tok.size, x.shape[1]), dtype=np.float64)
    for k in range(top_k):
        keep = (loc[:, k] >= 0)[:, None]
        routed += np.where(keep, w[:, k:k + 1].astype(np.float64) * f[:, k], 0.0)
    out = np.float64(rsf) * routed
    if shared_w13 is not None:
        for s in range(shared_w13.shape[0]):
            out += expert_mlp(x[tok], shared_w13[s], shared_w2[s])
    return out


def moe_forward_masked_loop(x, router_w, w13, w2, *, top_k, renormalize=True,
                            n_group=0, topk_group=0, rsf=1.0, router_b=None,
                            shared_w13=None, shared_w2=None, emap=None):
    """The page's dense form: every local expert runs on all tokens.

    MixtralMoE.forward loops over its expert indices. For each expert it forms
    the mask selected_experts == idx and the weight (routing_weights *
    mask).sum(-1). It runs the expert on all hidden states, scales by that
    weight and accumulates. Used only to pin ``moe_forward`` on small inputs.
    """
    ids, w, _ = route(x, router_w, router_b, top_k=top_k,
                      renormalize=renormalize, n_group=n_group,
                      topk_group=topk_group)
    E_l = w13.shape[0]
    if emap is None:
        emap = np.arange(E_l, dtype=np.int32)
    final = np.zeros((x.shape[0], x.shape[1]), dtype=np.float64)
    for g_id in np.nonzero(emap >= 0)[0]:
        e = emap[g_id]
        mask = ids == g_id
        ew = (w.astype(np.float64) * mask).sum(axis=-1, keepdims=True)
        final += expert_mlp(x, w13[e], w2[e]) * ew
    final *= np.float64(rsf)
    if shared_w13 is not None:
        for s in range(shared_w13.shape[0]):
            final += expert_mlp(x, shared_w13[s], shared_w2[s])
    return final


# ---------------------------------------------------------------------------
# token permutation by expert
# ---------------------------------------------------------------------------
def align_cap(T: int, top_k: int, n_local: int, block: int) -> int:
    """Rows needed for the padded permutation: T*K + E_local*(block-1)."""
    return T * top_k + n_local * (block - 1)


def align_permute(topk_ids, emap, n_local: int, block: int, cap=None):
    """Per-local-expert segments of work items, padded to ``block`` rows.

    Work item i = t*K + k stands for the pair (token t, slot k). This is the
    flattening in ep_fused_moe_patch.py, ``_ep_forward`` step 2, where
    ``flat_token_idx = arange(T)`` is expanded over K. Items whose expert is
    not local (emap = -1) are dropped (step 3 keeps only local ids). Reading
    taken where the page uses an unstable argsort: within a segment, items
    appear in ascending item order.

    Returns counts[E_l], offsets[E_l+1] (exclusive, padded), sorted_ids[cap]
    (sentinel T*K on padding) and inv_pos[T*K] (row of each item, -1 dropped).
    """
    ids = np.asarray(topk_ids)
    T, K = ids.shape
    n_items = T * K
    if cap is None:
        cap = align_cap(T, K, n_local, block)
    loc = local_slots(ids, emap).reshape(-1)
    counts = np.zeros(n_local, dtype=np.int32)
    offsets = np.zeros(n_local + 1, dtype=np.int32)
    sorted_ids = np.full(cap, n_items, dtype=np.int32)
    inv_pos = np.full(n_items, -1, dtype=np.int32)
    for e in range(n_local):
        items = np.nonzero(loc == e)[0]              # ascending item order
        counts[e] = items.size
        padded = -(-items.size // block) * block
        offsets[e + 1] = offsets[e] + padded
        sorted_ids[offsets[e]:offsets[e] + items.size] = items
        inv_pos[items] = offsets[e] + np.arange(items.size, dtype=np.int32)
    return counts, offsets, sorted_ids, inv_pos


def grouped_mlp(x, sorted_ids, offsets, w13, w2, top_k: int, rows=None):
    """y_perm[r] = f_e(x[sorted_ids[r] // K]) for each non-padding row r of
    segment e (fp64). Returns {row: vector} for ``rows`` (default: all)."""
    x = np.asarray(x)
    n_items = x.shape[0] * top_k
    E_l = w13.shape[0]
    seg = np.searchsorted(np.asarray(offsets), np.arange(len(sorted_ids)),
                          side="right") - 1
    want = np.arange(len(sorted_ids)) if rows is None else np.asarray(rows)
    out = {}
    for e in range(E_l):
        rs = [r for r in want if seg[r] == e and sorted_ids[r] < n_items]
        if rs:
            toks = np.asarray(sorted_ids)[rs] // top_k
            y = expert_mlp(x[toks], w13[e], w2[e])
            for j, r in enumerate(rs):
                out[int(r)] = y[j]
    return out


def combine(y_perm_rows, inv_pos, topk_w, rsf=1.0, shared_out=None):
    """out[t] = rsf * sum_k w[t,k] * y_perm[inv_pos[t,k]] + shared_out[t].

    This is the weighted gather back to token order. It is the same sum as the
    ``scatter_add_`` by token index in ep_fused_moe_patch.py ``_ep_forward``
    step 4, written per token. ``y_perm_rows`` is an array [cap, H]; rows with
    inv_pos = -1 are skipped.
    """
    w = np.asarray(topk_w, np.float64)
    T, K = w.shape
    y = np.asarray(y_perm_rows, np.float64)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    inv = np.asarray(inv_pos).reshape(T, K)
    for t in range(T):
        for k in range(K):
            r = inv[t, k]
            if r >= 0:
                out[t] += w[t, k] * y[r]
    out *= np.float64(rsf)
    if shared_out is not None:
        out += np.asarray(shared_out, np.float64)
    return out


def weight_bytes_per_card(n_experts, intermediate, hidden, n_layers, elem_bytes):
    """MoE weight bytes held by one card: experts * (2*I*H + H*I) * bytes * layers.

    The sizing formula of the ep_fused_moe_patch.py docstring ("Memory layout
    comparison").
    """
    per_expert = 2 * intermediate * hidden + hidden * intermediate
    return n_experts * per_expert * elem_bytes * n_layers


# ---------------------------------------------------------------------------
# expert-parallel dispatch and combine (the rank-local halves of the exchange)
# ---------------------------------------------------------------------------
def ep_dispatch(x, topk_ids, topk_w, num_experts, ep_size, pmap=None, n_local=None):
    """Send buffers of one rank, ordered by destination rank.

    ep_fused_moe_patch.py ``_ep_forward`` step 2: every (token, slot) work
    item goes to the rank owning its expert (dest = id // (E / ep_size)). Items
    are sorted by destination and (hidden row, weight, global id, token index)
    are packed, with per-destination counts for the all-to-all. The page sorts
    with ``argsort``, which leaves the order inside a destination open. Reading
    taken: a stable sort, so items keep ascending t*K + k order.

    With redundant experts (MoEMixin ``num_redundant_experts``: physical vs
    logical experts), ``pmap`` is the global replica map of ``physical_map``
    and ``n_local`` the weight slots per rank: an item goes to the replica
    ``physical_ids`` picks, dest = physical id // n_local, and the id sent is
    the physical one, so the receiver's local slot is id - rank * n_local.

    Returns (counts [ep] int64, send_pos [T*K] int32 = each item's row in the
    send buffer, send_x [T*K, H], send_ids [T*K] int32, send_w [T*K] fp32,
    send_tok [T*K] int32).
    """
    T, K = np.asarray(topk_ids).shape
    if pmap is None:
        ids = np.asarray(topk_ids).reshape(-1)
        n_local = num_experts // ep_size
    else:
        ids = physical_ids(topk_ids, pmap).reshape(-1)
    w = np.asarray(topk_w, np.float32).reshape(-1)
    dest = ids // n_local
    order = np.argsort(dest, kind="stable")
    counts = np.bincount(dest, minlength=ep_size).astype(np.int64)
    send_pos = np.empty(T * K, dtype=np.int32)
    send_pos[order] = np.arange(T * K, dtype=np.int32)
    tok = order // K
    return (counts, send_pos, np.asarray(x)[tok], ids[order].astype(np.int32),
            w[order], tok.astype(np.int32))


def ep_expert_compute(recv_x, recv_ids, recv_w, w13_local, w2_local, start_expert):
    """Rows a rank sends back for the items it received, fp64.

    ``_ep_forward`` step 3: local id = global id - start_expert, and the local
    experts run with top_k = 1 per received item. The page passes the item's
    weight to ``fused_experts``, so each returned row is already weighted:
    y[r] = w[r] * f_{id[r] - start}(x[r]).
    """
    rx = np.asarray(recv_x, np.float64)
    lid = np.asarray(recv_ids) - start_expert
    y = np.zeros_like(rx)
    for e in np.unique(lid):
        rows = np.nonzero(lid == e)[0]
        y[rows] = expert_mlp(rx[rows], w13_local[e], w2_local[e])
    return y * np.asarray(recv_w, np.float64)[:, None]


def ep_combine(ret_rows, send_pos, top_k, rsf=1.0, shared_out=None):
    """out[t] = rsf * sum_k ret[send_pos[t*K + k]] + shared_out[t].

    ``_ep_forward`` step 4: the returned rows come back in send order. They
    are un-sorted and scatter-added by token index, unweighted because the
    weights were applied by the expert-holding rank. rsf and the shared
    experts then apply as in the single-rank forward.
    """
    ret = np.asarray(ret_rows, np.float64)
    pos = np.asarray(send_pos).reshape(-1, top_k)
    out = np.zeros((pos.shape[0], ret.shape[1]), dtype=np.float64)
    for k in range(top_k):
        out += ret[pos[:, k]]
    out *= np.float64(rsf)
    if shared_out is not None:
        out += np.asarray(shared_out, np.float64)
    return out


def ep_exchange(send_bufs, send_counts):
    """All-to-all of per-rank send buffers (host simulation of the exchange).

    send_bufs[r] is rank r's buffer ordered by destination and
    send_counts[r][d] the number of its rows for rank d. Rank d receives the
    rows for it from every rank, concatenated in source-rank order, as
    ``all_to_all_single`` with split sizes does.
    """
    ep = len(send_bufs)
    offs = [np.concatenate([[0], np.cumsum(c)]) for c in send_counts]
    return [np.concatenate([send_bufs[s][offs[s][d]:offs[s][d + 1]] for s in range(ep)])
            for d in range(ep)]
