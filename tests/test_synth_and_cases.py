"""The seeded input generator and the gap-checked case builder (CPU only)."""
import numpy as np

import synth
from oracle import cases, moe_oracle as O


def test_rows_are_independent_streams():
    a = synth.draw(0, synth.W13, 0, 10, 33, 1.0, True)
    b = synth.draw(0, synth.W13, 4, 3, 33, 1.0, True)
    np.testing.assert_array_equal(a[4:7], b)
    c = synth.draw(1, synth.W13, 0, 10, 33, 1.0, True)
    assert not np.array_equal(a, c)


def test_bf16_values_are_exact_and_bits_agree():
    a = synth.draw(5, synth.X, 0, 64, 128, 0.3, True)
    bits = synth.draw_bf16_bits(5, synth.X, 0, 64, 128, 0.3)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(bits), a)
    low = a.view(np.uint32) & 0xFFFF
    assert (low == 0).all()


def test_normal_moments():
    z = synth.draw(9, synth.X, 0, 512, 1024, 2.0, False).astype(np.float64)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 2.0) < 0.01
    assert abs(((z / 2.0) ** 4).mean() - 3.0) < 0.05


def test_ep_shard_is_slice_of_global():
    wl = synth.EP_SHARD.with_(H=64, I=32, E=16, ep_size=4, ep_rank=2, T=4)
    loc = synth.draw_tensor(wl, synth.W13)
    glob = synth.draw_tensor(wl, synth.W13, local=False)
    np.testing.assert_array_equal(loc, glob[8:12])
    loc2 = synth.draw_tensor(wl, synth.W2)
    np.testing.assert_array_equal(loc2, synth.draw_tensor(wl, synth.W2, local=False)[8:12])


def test_attempts_redraw_only_that_row():
    att = np.zeros(6, np.int32)
    a = synth.draw(0, synth.X, 0, 6, 16, 1.0, True, att)
    att[3] = 2
    b = synth.draw(0, synth.X, 0, 6, 16, 1.0, True, att)
    np.testing.assert_array_equal(np.delete(a, 3, 0), np.delete(b, 3, 0))
    assert not np.array_equal(a[3], b[3])


def test_gap_checked_case_tiny_and_decode():
    for wl in (synth.TINY, synth.QWEN_DECODE.with_(T=64, H=256, I=64),
               synth.DEEPSEEK.with_(T=48, H=256, I=128, I_shared=128)):
        d = cases.build_case(wl)
        gap = O.routing_min_gap(d["p"], wl.K, wl.n_group, wl.topk_group)
        assert gap.min() >= cases.MIN_GAP
        d2 = cases.build_case(wl)
        np.testing.assert_array_equal(d["x"], d2["x"])
        np.testing.assert_array_equal(d["attempts"], d2["attempts"])
