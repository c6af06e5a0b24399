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


def test_single_core_oracle_figures(oracle_mod):
    out = bench._oracle_single_core(budget_s=0.05)
    for name in ("tiny", "tiny_causal", "b4h12_q1000_k4097_d64_cross"):
        assert out[name] > 0, out
    assert "one thread" in out["sample"]
