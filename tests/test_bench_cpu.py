"""The bench's host-side helpers, on the CPU: the distinct-expert count behind
the bytes roofline, the peaks it divides by, the profiled-traffic lookups
(per hot expert for decode calls, per routed pick for prefill calls), the
workload table and the library's prefill tile widths."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench                                # noqa: E402
import synth                                # noqa: E402


def test_distinct_experts_counts_each_expert_once_per_bank():
    mask = np.array([1, 1, 0, 1, 0, 0], np.uint8)       # experts 0, 1, 3 hot; 2, 4, 5 cold
    ids = np.array([[0, 2], [0, 4], [1, 2], [2, 0]])    # hot {0, 1}, cold {2, 4}
    assert bench.distinct_experts(ids, mask) == (2, 2)
    assert bench.distinct_experts(np.array([[3, 3]]), mask) == (1, 0)


def test_bytes_roofline_terms_match_the_expert_size():
    # the bench's per-expert bytes are the library's and the oracle's byte model
    cfg = synth.get_config("decode1")
    assert synth.expert_bytes(cfg.H, cfg.I) == 18_800_640


def test_peaks_are_positive_and_labelled():
    hbm, burst, sustained, src = bench.load_peaks()
    assert hbm > 1000 and burst > 100 and 0 < sustained <= burst * 1.2
    assert src in ("measured", "fallback")
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        assert src == "measured" and hbm == float(json.load(open(p))["hbm_gbs"])


def test_profiled_traffic_only_for_the_profiled_source():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["decode1"]
    got = bench.profiled_traffic("decode1")
    if rec["source_sha"] == bench.source_sha():
        assert got == rec["bytes_per_hot_expert"]
        # a hot expert's DRAM bytes within a few percent of its algorithmic bytes
        assert 1.0 <= got / 18_800_640 <= 1.05
    else:
        assert got is None
    assert bench.profiled_traffic("no-such-workload") is None


def test_every_workload_is_a_generator_config():
    for name in bench.WORKLOADS:
        cfg = synth.get_config(name)
        assert cfg.E == 384 and cfg.k == 6 and cfg.H == 4096 and cfg.I == 2880


def test_prefill_traffic_is_per_routed_pick_of_the_profiled_source():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for name in ("prefill", "prefill_mxfp8"):
        rec = d[name]
        got = bench.profiled_traffic(name, "bytes_per_pick")
        if rec["source_sha"] != bench.source_sha():
            assert got is None
            continue
        # the per-launch reads and writes add up to the captured step, and the
        # per-pick figure is that over the captured picks
        tot = sum(rec["dram_read_bytes"].values()) + sum(rec["dram_write_bytes"].values())
        assert tot == rec["dram_bytes_captured_step"]
        assert got == round(tot / rec["picks_captured_step"])
        # a pick's share of the weights at about 128 picks per expert, within
        # the rows it adds: 18.8 MB / 128 = 147 KB plus at most ~80 KB of rows
        assert 140e3 < got < 230e3


def test_prefill_tile_widths_match_the_library():
    # the shifted-prefill link-byte accounting counts tiles with the library's
    # token-tile widths; read them from the library's source
    import re
    src = open(os.path.join(ROOT, "cold_expert_residency_gb300", "csrc", "moe_internal.cuh")).read()
    two = int(re.search(r"constexpr int kPrefillTile = (\d+);", src).group(1))
    mx = int(re.search(r"constexpr int kPrefillTileMx = (\d+);", src).group(1))
    assert (bench.kPrefillTile, bench.kPrefillTileMx) == (two, mx)


def test_bytes_roofline_on_a_hand_example():
    # two steps of two layers; an expert of 1e9 bytes, HBM 1000 GB/s (1 ms per
    # expert), link 100 GB/s (10 ms per expert)
    dh = [[3, 2], [1, 0]]
    dc = [[0, 1], [1, 0]]
    r = bench.bytes_roofline(dh, dc, [40.0, 20.0], 1e9, 1000.0, 100.0)
    # per layer-step: max(hot, cold) = 3, 10, 10, 0 ms; sums 3, 12, 11, 0 ms
    assert abs(r["frac_max"] - 23.0 / 60.0) < 1e-12
    assert abs(r["frac_sum"] - 26.0 / 60.0) < 1e-12
    assert abs(r["t_roof_max_us"] - 11.5e3) < 1e-6 and abs(r["t_roof_sum_us"] - 13.0e3) < 1e-6
    assert abs(r["t_step_us"] - 30.0e3) < 1e-6
    assert r["distinct_hot"] == 3.0 and r["distinct_cold"] == 1.0
    # the max form never exceeds the sum form
    assert r["frac_max"] <= r["frac_sum"]


def test_ffn_roofline_and_whole_job_rate():
    import types
    S = types.SimpleNamespace(hbm_peak=5000.0, peak_src="measured")
    r = bench.ffn_roofline(S, "k", [10, 30], [2.0, 2.0], 1e8, traffic_per_expert=1.01e8)
    # 20 experts of 0.1 GB in 2 ms: 1000 GB/s, 0.2 of the peak; traffic 20 x 1.01e8
    assert abs(r["achieved"] - 1000.0) < 1e-9 and abs(r["frac"] - 0.2) < 1e-12
    assert abs(r["traffic"] - 2.02e9) < 1e-3 and r["algorithmic_bytes"] == 2e9
    assert bench.ffn_roofline(S, "k", [10], [1.0], 1e8)["traffic"] is None
    # 2 ranks x 112 tokens x 10 steps over the slowest rank's 70 ms
    assert abs(bench.job_tokens_per_s(2, 112, 10, 70.0) - 32000.0) < 1e-9


def test_profile_key_ignores_comments_but_not_code():
    src = 'int f(int a) {  // the first\n  /* two\n lines */ return a + 1; }\nconst char *s = "x // y";\n'
    same = '// a header\nint f(int a)\n{\n    return a + 1;  /* once */\n}\nconst char *s = "x // y";'
    assert bench.code_only(src) == bench.code_only(same)
    assert bench.code_only(src) != bench.code_only(src.replace("a + 1", "a + 2"))
    # text inside a string literal is code, even when it looks like a comment
    assert bench.code_only(src) != bench.code_only(src.replace('"x // y"', '"x // z"'))
    assert bench.code_only("char c = '/'; // c\nint d;") == "char c = '/'; int d;"
