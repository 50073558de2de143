"""Host-side pieces of bench.py that need no GPU: the clock record summary,
the DRAM-traffic lookup from the committed ncu summaries, and the rules
those summaries follow (every ncu command leaves the clocks alone)."""
import hashlib
import json
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _row(sm, mx, power_cap="Not Active", hw="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return f"0, {sm}, {mx}, 1210.50, 0x0000000000000004, {hw}, Not Active, Not Active, {power_cap}"


def test_clock_summary_takes_median_max_and_every_active_reason():
    lines = [_row(1785, 2070), _row(1800, 2070, power_cap="Active"), _row(1900, 2070),
             "0, [N/A], [N/A], [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage", ""]
    s = bench.summarize_clocks(lines)
    assert s == {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
    s = bench.summarize_clocks([_row(2070, 2070, hw="Active"), _row(2070, 2070)])
    assert s["reasons"] == ["hw_slowdown"] and s["sm_mhz"] == 2070.0
    assert bench.summarize_clocks(["garbage"]) is None


def test_traffic_lookup_follows_the_kernel_source_hash(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("// kernel v1\n")
    (tmp_path / "profiles").mkdir()
    entry = {"kernel": "k", "kernel_source": "k.cu",
             "kernel_sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
             "dram_bytes_per_launch": 12345}
    (tmp_path / "profiles" / "dominant_kernel_traffic.json").write_text(
        json.dumps({"workloads": {"w": entry}}))
    assert bench.traffic_from_profile("w", "k.cu", root=str(tmp_path)) == 12345
    assert bench.traffic_from_profile("other", "k.cu", root=str(tmp_path)) is None
    assert bench.traffic_from_profile("w", "j.cu", root=str(tmp_path)) is None
    src.write_text("// kernel v2\n")  # the kernel changed since the capture
    assert bench.traffic_from_profile("w", "k.cu", root=str(tmp_path)) is None


def test_committed_profiles_name_existing_sources_and_leave_clocks_alone():
    with open(os.path.join(ROOT, "profiles", "dominant_kernel_traffic.json")) as fh:
        d = json.load(fh)
    assert d["workloads"]
    for name, v in d["workloads"].items():
        assert os.path.exists(os.path.join(ROOT, v["kernel_source"])), name
        assert re.fullmatch(r"[0-9a-f]{64}", v["kernel_sha256"]), name
        assert v["dram_bytes_per_launch"] > 0, name
        assert v["command"].startswith("ncu ") and "--clock-control none" in v["command"]
        assert "bench.py" in v["command"] and "_work" not in v["command"]
    for fn in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        if not fn.endswith(".md"):
            continue
        text = open(os.path.join(ROOT, "profiles", fn)).read()
        for cmd in re.findall(r"^ncu [^\n]*(?:\\\n[^\n]*)*", text, flags=re.M):
            assert "--clock-control none" in cmd, (fn, cmd)


def test_tensor_bound_roofline_takes_the_burst_peak():
    """The dominant kernel runs inside a timed region of milliseconds, so a
    tensor-bound fraction is taken against the burst bf16 peak; the sustained
    fraction is a secondary key. An HBM-bound kernel is taken against the copy
    peak. GEMM1 on CTA pairs reads the permuted rows (one per assignment); on
    single CTAs it gathers from x, each distinct token row counted once."""
    import synth

    class Plan:
        fused_mlp, cta_pairs = 0, 1

    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0,
             "source": "measured"}
    wl = synth.MIXTRAL
    A, touched = 8192, 8
    flops = 4 * A * wl.H * wl.I
    k_ms = flops / 1.5e15 * 1e3          # 1500 TFLOP/s
    r = bench.dominant_kernel_roofline(wl, Plan, A, touched, 4096, k_ms, peaks)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0
    assert abs(r["frac"] - 0.75) < 1e-3 and abs(r["frac_of_sustained"] - 0.9375) < 1e-3

    class Fused:
        fused_mlp, cta_pairs = 1, 0

    wl = synth.QWEN_DECODE.with_(T=8)
    A, touched = 64, 36
    r = bench.dominant_kernel_roofline(wl, Fused, A, touched, 8, 0.05, peaks)
    assert r["bound"] == "hbm" and r["peak"] == 6000.0
    want = (touched * 3 * wl.H * wl.I * 2 + (2 * A * wl.H + 2 * A * wl.I) * 2) / 0.05e-3 / 1e9
    assert abs(r["achieved"] - want) < 0.1

    class Single:
        fused_mlp, cta_pairs = 0, 0

    wl = synth.EP_SHARD
    A, touched, rows = 16384, 64, 7400
    r = bench.dominant_kernel_roofline(wl, Single, A, touched, rows, 0.1, peaks)
    assert r["bound"] == "hbm"
    assert r["algorithmic_bytes"] == (touched * 2 * wl.I * wl.H + rows * wl.H + A * wl.I) * 2
    r = bench.dominant_kernel_roofline(wl, Plan, A, touched, rows, 0.1, peaks)
    assert r["algorithmic_bytes"] == (touched * 2 * wl.I * wl.H + A * wl.H + A * wl.I) * 2


def test_layer_roofline_and_extra_workload_list():
    import synth
    wl = synth.QWEN_DECODE.with_(T=8)
    flops, nbytes = bench.layer_work(wl, 64, 36)
    assert nbytes == 36 * 3 * 2048 * 512 * 2 + 256 * 2048 * 2 + 2 * 8 * 2048 * 2
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    r = bench.layer_roofline(flops, nbytes, 0.05, peaks)
    assert abs(r["frac_of_hbm"] - nbytes / 0.05e-3 / 6e12) < 1e-4
    # every configured workload except the tiny parity case is timed in one run,
    # the decode sizes last with the largest T (whose weights they share) last
    names = set(bench.EXTRA_WORKLOADS)
    assert names == {n for n in bench.WORKLOADS if n != "tiny"}
    dec = [n for n in bench.EXTRA_WORKLOADS if n.startswith("qwen3_decode_T")]
    assert bench.EXTRA_WORKLOADS[-len(dec):] == dec
    assert dec[-1] == f"qwen3_decode_T{max(synth.DECODE_TOKENS)}"
