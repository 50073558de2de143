"""moe_align_permute_noalloc against moe_align_permute, through the C ABI.

The no-allocation variant serves callers that cannot hand the library a
workspace: hosts whose own memory pool owns all device memory, serving loops
that cannot afford cudaMalloc's implicit synchronisation, and fixed-budget
embedded callers. Its scratch is a static device array shared by every call.
The test makes two calls in a row with different shapes, so the second one
runs over the first one's leftover scratch. Each result must equal the
workspace entry point's exactly (these are integer outputs). A size beyond
the array must be refused.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from expert_moe_layer_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _ids(T, K, E, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


def _run(fn, cfg, T, ids, block, emap=None):
    El = cfg.num_experts // cfg.ep_size
    cap = B.align_cap(cfg, T, block)
    d_ids = torch.from_numpy(ids).cuda()
    em = None if emap is None else torch.from_numpy(emap).cuda()
    counts = torch.full((El,), -5, dtype=torch.int32, device="cuda")
    offsets = torch.full((El + 1,), -5, dtype=torch.int32, device="cuda")
    sorted_ids = torch.full((cap,), -5, dtype=torch.int32, device="cuda")
    inv_pos = torch.full((T * cfg.top_k,), -5, dtype=torch.int32, device="cuda")
    if fn == "noalloc":
        B.moe_align_permute_noalloc(cfg, T, d_ids, em, block, counts, offsets, sorted_ids,
                                    inv_pos, cap)
    else:
        ws = torch.empty(B.align_workspace_size(cfg, T), dtype=torch.uint8, device="cuda")
        B.moe_align_permute(cfg, T, d_ids, em, block, counts, offsets, sorted_ids, inv_pos,
                            cap, ws)
        assert B.moe_get_status(ws) == (0, 0)
    torch.cuda.synchronize()
    return [a.cpu().numpy() for a in (counts, offsets, sorted_ids, inv_pos)]


CALLS = [
    # (E, K, ep_size, ep_rank, T, block): a large shard first, then a smaller one
    (256, 8, 4, 1, 8192, 16),
    (160, 6, 1, 0, 777, 7),
]


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    for i, (E, K, ep, r, T, block) in enumerate(CALLS):
        cfg = B.make_config(E, K, 2048, 512, ep_size=ep, ep_rank=r)
        ids = _ids(T, K, E, seed=100 + i)
        want = _run("ws", cfg, T, ids, block)
        got = _run("noalloc", cfg, T, ids, block)
        for name, a, b in zip(("counts", "offsets", "sorted_ids", "inv_pos"), got, want):
            np.testing.assert_array_equal(a, b, err_msg=f"call {i}: {name}")


def test_noalloc_with_expert_map_repeated():
    E, K, T = 64, 4, 3000
    cfg = B.make_config(E, K, 1024, 512, ep_size=2, ep_rank=0)
    rng = np.random.default_rng(3)
    emap = np.full(E, -1, dtype=np.int32)
    emap[rng.choice(E, E // 2, replace=False)] = rng.permutation(E // 2).astype(np.int32)
    ids = _ids(T, K, E, seed=9)
    want = _run("ws", cfg, T, ids, 16, emap)
    for _ in range(2):
        got = _run("noalloc", cfg, T, ids, 16, emap)
        for a, b in zip(got, want):
            np.testing.assert_array_equal(a, b)


def test_noalloc_refuses_sizes_beyond_its_static_scratch():
    cfg = B.make_config(256, 8, 2048, 512)
    T = 65536                       # 2048 warps x 256 experts of counts > 1 MiB
    assert B.align_workspace_size(cfg, T) > (1 << 20)
    small = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as err:
        B.moe_align_permute_noalloc(cfg, T, small, None, 16, small, small, small, small,
                                    B.align_cap(cfg, T, 16))
    assert err.value.status == 3    # MOE_ERR_WORKSPACE
    assert (small == 0).all()
