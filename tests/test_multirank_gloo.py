"""The multi-rank paths on CPU: world_size 2 over gloo.

Expert parallelism splits a layer by experts. Each rank computes the partial
output of its local experts for all tokens, and one exchange sums the partials
(ep_fused_moe_patch.py, _ep_forward: global routing, local compute, results
back to the tokens; vllm-omni "Expert Parallel": allgather/reducescatter
backend). Here the ranks are CPU processes, each rank's partial comes from
the oracle, and the exchange is a gloo all-reduce. The sum must equal the
unsharded layer. The second test covers bench.py's aggregation of replicas:
the slowest rank's time and the tokens of all ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _layer(seed=5, T=12, H=16, I=8, E=8, S=1):
    r = np.random.default_rng(seed)
    return dict(x=r.standard_normal((T, H)), router_w=r.standard_normal((E, H)) * 0.5,
                w13=r.standard_normal((E, 2 * I, H)) / 4, w2=r.standard_normal((E, H, I)) / 3,
                shared_w13=r.standard_normal((S, 2 * I, H)) / 4,
                shared_w2=r.standard_normal((S, H, I)) / 3)


def _ep_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import moe_oracle as O
    _init(rank, world, port)
    d = _layer()
    E = d["w13"].shape[0]
    El = E // world
    emap = O.expert_map(E, world, rank)
    part = O.moe_forward(d["x"], d["router_w"], d["w13"][rank * El:(rank + 1) * El],
                         d["w2"][rank * El:(rank + 1) * El], top_k=3, renormalize=True,
                         rsf=2.0, emap=emap,
                         shared_w13=d["shared_w13"] if rank == 0 else None,
                         shared_w2=d["shared_w2"] if rank == 0 else None)
    t = torch.from_numpy(part)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    if rank == 0:
        full = O.moe_forward(d["x"], d["router_w"], d["w13"], d["w2"], top_k=3,
                             renormalize=True, rsf=2.0, shared_w13=d["shared_w13"],
                             shared_w2=d["shared_w2"])
        q.put(float(np.abs(t.numpy() - full).max()))
    dist.destroy_process_group()


def _a2a(buf, send_counts, recv_counts):
    """all_to_all_single of the rows of a numpy buffer with split sizes."""
    t = torch.from_numpy(np.ascontiguousarray(buf))
    out = torch.empty((int(sum(recv_counts)),) + tuple(t.shape[1:]), dtype=t.dtype)
    dist.all_to_all_single(out, t, output_split_sizes=[int(c) for c in recv_counts],
                           input_split_sizes=[int(c) for c in send_counts])
    return out.numpy()


def _ep_dispatch_worker(rank, world, port, q):
    """The page's _ep_forward on real ranks: every rank routes its own tokens
    over all experts, all-gathers the send counts, exchanges (rows, ids,
    weights) with all_to_all_single, runs its expert shard on what it
    received, sends the rows back and combines. The exchange logic around
    the library's dispatch/compute/combine calls is checked here, with the
    oracle standing in for them."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import moe_oracle as O
    _init(rank, world, port)
    d = _layer()
    E = d["w13"].shape[0]
    El = E // world
    x = np.random.default_rng(40 + rank).standard_normal(((9, 4)[rank], d["x"].shape[1]))
    ids, w, _ = O.route(x, d["router_w"], top_k=3, renormalize=True)
    counts, pos, sx, sids, sw, _ = O.ep_dispatch(x, ids, w, E, world)
    parts = [torch.zeros(world, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(parts, torch.from_numpy(counts))
    recv_counts = [int(p[rank]) for p in parts]
    rx = _a2a(sx, counts, recv_counts)
    rids = _a2a(sids, counts, recv_counts)
    rw = _a2a(sw, counts, recv_counts)
    y = O.ep_expert_compute(rx, rids, rw, d["w13"][rank * El:(rank + 1) * El],
                            d["w2"][rank * El:(rank + 1) * El], rank * El)
    ret = _a2a(y, recv_counts, counts)
    out = O.ep_combine(ret, pos, 3, rsf=2.0)
    full = O.moe_forward(x, d["router_w"], d["w13"], d["w2"], top_k=3, renormalize=True,
                         rsf=2.0)
    q.put(float(np.abs(out - full).max()))
    dist.destroy_process_group()


def _bench_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    _init(rank, world, port)
    local_ms = [100.0, 250.0][rank]          # rank 1 is slower
    total, tps = bench.aggregate_over_ranks(local_ms, tokens_per_rank=4096, steps=10,
                                            world=world)
    q.put((rank, total, tps))
    dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=fn, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    return [q.get(timeout=5) for _ in range(q.qsize())] if hasattr(q, "qsize") else []


def test_ep_partial_outputs_all_reduce_to_unsharded_layer():
    out = _run(_ep_worker)
    assert len(out) == 1 and out[0] < 1e-12


def test_ep_dispatch_all_to_all_equals_unsharded_layer():
    out = _run(_ep_dispatch_worker)
    assert len(out) == 2 and max(out) < 1e-12


def test_bench_aggregates_slowest_rank_and_all_tokens():
    out = sorted(_run(_bench_worker))
    assert len(out) == 2
    for _, total, tps in out:
        assert total == 250.0
        assert tps == pytest.approx(2 * 4096 * 10 / 0.25)
