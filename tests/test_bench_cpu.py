"""Host-side parts of the benchmark that run without a GPU: the sizing of the reference
arm's oracle sample and the one-thread oracle figures that the CPU baseline reports."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_run_is_bounded_for_any_step_count():
    for steps, warmup in ((1, 3), (2, 3), (50, 5), (2000, 10), (100000, 10)):
        per = bench.reference_step_budget(steps, warmup)
        assert 0 < per <= 10.0
        assert per * (steps + warmup) <= 100.0 + 1e-9
    assert bench.reference_step_budget(2, 3) == 10.0


def test_whole_config_oracle_figures(oracle_mod):
    """Whole configurations timed end to end on all threads and, where asked, on one (the
    small ones here; the bench adds the d=64 cross-attention and the two benchmark
    workloads)."""
    out = bench._oracle_whole_configs(configs=(("tiny", True), ("tiny_causal", False)))
    for label in ("all_threads", "one_thread"):
        r = out["tiny"][label]
        assert r["ms"] > 0 and r["tflops"] > 0, out
    assert out["tiny"]["one_thread"]["threads"] == 1
    assert set(out["tiny_causal"]) == {"all_threads"}
    assert "whole configurations" in out["note"]
    names = [n for n, _ in bench.WHOLE_CONFIGS]
    assert {"tiny", "tiny_causal", "b4h12_q1000_k4097_d64_cross", "b2h8_n4096_d128_full",
            "b2h8_n8192_d128_causal"} == set(names)


def test_failed_side_run_is_reported_not_raised(monkeypatch):
    import subprocess
    import types

    calls = []

    def fake_run(cmd, **kw):
        calls.append(cmd)
        if "--bwd" in cmd:
            raise subprocess.TimeoutExpired(cmd, 600)
        if "--fp8" in cmd:
            return types.SimpleNamespace(stdout="", stderr="boom", returncode=1)
        line = ('{"value": 1.5, "unit": "TFLOPS", "config": {"entry_point": "fa_fwd"}, '
                '"breakdown": {"w": {"ms": 0.1, "tflops": 1.5, "pct_of_peak": 0.1}}}')
        return types.SimpleNamespace(stdout="noise\n" + line + "\n", stderr="", returncode=0)

    monkeypatch.setattr(subprocess, "run", fake_run)
    args = types.SimpleNamespace(steps=2000)
    out = bench.secondary_measurements(args)
    assert len(calls) == len(out)
    assert "error" in out["bwd"] and "TimeoutExpired" in out["bwd"]["error"]
    assert "error" in out["fwd_fp8_e4m3"]
    ok = out["fwd_tiny_full_and_causal"]
    assert ok["value"] == 1.5 and ok["breakdown"]["w"]["pct_of_peak"] == 0.1
    for cmd in calls:  # every side run is a bounded, single-purpose bench process
        assert "--no-also" in cmd and "--cpu-budget" in cmd
        assert cmd[cmd.index("--steps") + 1] == "100"


def test_visible_scores_and_sfu_bound():
    """The exponential count of the secondary bound: one per (row, visible key), causal rows
    seeing keys j <= i; and the bound's arithmetic."""
    import bench
    import gen
    w = gen.WORKLOADS["b2h8_n8192_d128_causal"]
    assert bench.visible_scores(w) == 2 * 8 * 8192 * 8193 // 2
    w = gen.WORKLOADS["b4h12_q1000_k4097_d64_cross"]
    assert bench.visible_scores(w) == 4 * 12 * 1000 * 4097
    w = gen.custom(1, 2, 10, 4, 64, gen.BF16, True)  # rows 3..9 see all 4 keys
    assert bench.visible_scores(w) == 2 * (1 + 2 + 3 + 4 * 7)
    w = gen.custom(1, 1, 3, 10, 64, gen.BF16, True)  # Nq < Nk: rows see 1, 2, 3 keys
    assert bench.visible_scores(w) == 6
    b = bench.sfu_bound(gen.WORKLOADS["b2h8_n8192_d128_causal"], ms=0.2, sms=152, sm_mhz=2000.0)
    assert b["peak_ex2_per_s"] == 32 * 152 * 2000e6
    assert abs(b["achieved_ex2_per_s"] - b["ex2_count"] / 0.2e-3) < 1
    assert "xu_inst_counted" not in b
    b = bench.sfu_bound(gen.WORKLOADS["b2h8_n8192_d128_causal"], ms=0.2, sms=152, sm_mhz=2000.0,
                        counters={"xu_inst": b["ex2_count"] // 32 * 103 // 100})
    assert b["xu_inst_per_ex2_warp_inst"] == 1.03


def test_recorded_counters_match_source_and_entry():
    """The committed ncu record is used only for the kernel source it was taken on and for
    the entry point it was taken through; its XU count covers the ex2s the scores need."""
    import json
    import bench
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    for name, k in rec["kernels"].items():
        assert k["dram_bytes_per_launch"] == k["read"] + k["write"]
        assert 1.0 <= k["xu_inst"] / k["ex2_warp_inst"] < 1.1, name
        if rec["source_sha256"] == bench.kernel_source_hash():
            assert bench.recorded_counters(name, k["entry"]) == k
            other = "fa_fwd" if k["entry"] == "fa_fwd_ws" else "fa_fwd_ws"
            assert bench.recorded_counters(name, other) is None
