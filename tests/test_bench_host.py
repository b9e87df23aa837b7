"""Host-side logic of bench.py (no GPU): the FLOP formulas, the whole-job
aggregate at one rank, the DRAM-traffic table's source-digest gate, and the
parsing of the nvidia-smi clock samples that decide whether a run is kept."""
import math

import bench
import workloads as W


def test_flop_formulas():
    w = W.WORKLOADS["gpt2_small"]                      # causal: half of 4 B H N^2 d
    f, b = bench.flops(w)
    assert f == 4 * 8 * 12 * 1024 ** 2 * 64 / 2 and b == 2.5 * f
    w = W.WORKLOADS["long_n4096_noncausal"]
    f, b = bench.flops(w)
    assert f == 4 * 16 * 4096 ** 2 * 128 and b == 2.5 * f


def test_effective_flops_count_visible_keys_only():
    import torch
    w = W.WORKLOADS["bert_large"].with_(B=3)
    kv = torch.tensor([256, 512, 700], dtype=torch.int32)   # 700 is clamped to N = 512
    f, b = bench.effective_flops(w, kv)
    assert f == sum(4.0 * w.H * w.N * n * w.d for n in (256, 512, 512)) and b == 2.5 * f
    nominal, _ = bench.flops(w)
    assert f < nominal


def test_whole_job_aggregate_single_rank():
    value, ms = bench.whole_job_tflops(1, 2.0e12, 4.0)
    assert ms == 4.0 and math.isclose(value, 2.0e12 / 4.0e-3 / 1e12)


def test_traffic_reported_only_for_unchanged_sources(monkeypatch):
    digest = bench.source_digest("fa_fwd_kernel.cuh")
    assert digest is not None and len(digest) == 16
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {
        ("fwd", "a"): (123, "fa_fwd_kernel.cuh", digest),
        ("fwd", "b"): (456, "fa_fwd_kernel.cuh", "0" * 16),
        ("fwd", "c"): (789, "no_such_file.cuh", digest)})
    assert bench.ncu_traffic("fwd", "a") == 123
    assert bench.ncu_traffic("fwd", "b") is None      # captured from other sources
    assert bench.ncu_traffic("fwd", "c") is None
    assert bench.ncu_traffic("fwd", "missing") is None


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.proc = _DoneProc()
    s.lines = lines
    return s


def test_clock_samples_median_and_reasons():
    row = "0, {sm}, 2070, 950.2, {act}, Not Active, Not Active, Not Active, {cap}"
    lines = [(1.0, row.format(sm=2070, act="Active", cap="Active")),
             (1.2, row.format(sm=1980, act="Not Active", cap="Not Active")),
             (1.4, row.format(sm=2070, act="Not Active", cap="Not Active")),
             (1.6, "garbage line"),
             (9.0, "0, 100, 2070, 10, Active, Active, Not Active, Not Active, Not Active")]
    out = _sampler(lines).stop(window=(0.9, 1.7))      # the sample at t = 9 is outside
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    out = _sampler(lines).stop()                        # no window: every sample counts
    assert out["samples"] == 4 and "hw_slowdown" in out["reasons"]


def test_clock_sampler_without_nvidia_smi():
    out = bench.ClockSampler(0).stop()
    assert out["sm_mhz"] is None and out["reasons"] == ["nvidia-smi unavailable"]
