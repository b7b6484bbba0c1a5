"""bench.py's host-side logic on the CPU: the roofline numerators (a launch's and a round's algorithmic bytes)
from hand-worked trees, the launch count, the peaks' fallback, and the rule that a committed ncu traffic figure
counts only while the call's sources are the ones it was taken on, and the SM-clock sampler against a fake NVML
(read-only queries: median clock, throttle reasons, no library)."""
import json
import os

import numpy as np

import bench
from speculative_decoding_tree_top_gb300 import synth


def shape(**kw):
    base = dict(B=2, V=1000, K=4, M=8, H=16, E=24, n=4, max_depth=3, T=0.0, dtype="bf16", logit_scale=1.0,
                boost_count=0, boost_lo=0.0, boost_hi=0.0, name="hand")
    base.update(kw)
    return synth.Shape(**base)


def test_algorithmic_bytes_of_hand_worked_trees():
    s = shape()
    # request 0 pops depths 1, 1, 2, 3: the first n - 1 = 3 pops are expanded (all below the depth limit 3), into
    # positions 1, 1, 2, and the root into position 0 -> positions {0, 1, 2}, 3 GRU steps;
    # request 1 pops depths 1, 2, 3, 3: pops 0 and 1 are expanded (the third sits at the limit) -> {0, 1, 2}, 2 steps
    depth = np.array([[1, 1, 2, 3], [1, 2, 3, 3]])
    tokens = np.zeros((2, 4), np.int32)
    parents = np.array([[-1, -1, 0, 2], [-1, 0, 1, 1]])
    topm, build, parts = bench.algorithmic_bytes(s, tokens, parents, depth)
    assert parts["w_c_rows"] == (3 + 3) * 8 * 16 * 2          # M rows of H bf16 per expanded position
    assert parts["emb_rows"] == (3 + 2) * 24 * 2              # one embedding row of E bf16 per GRU step
    assert parts["gru_weights"] == 3 * 16 * (24 + 16) * 2 + 6 * 16 * 2
    assert topm == 2 * 4 * 1000 * 2 + 2 * 4 * 8 * 8           # the logits once, ids and values written
    # plus the top-M ids/values and h0 read, the tree (16 bytes a node, n x n mask) written
    assert build == parts["w_c_rows"] + parts["emb_rows"] + parts["gru_weights"] + 512 + 2 * 16 * 4 + 2 * 4 * 16 + 2 * 16
    assert bench.round_bytes(s, parts) == 2 * 4 * 1000 * 2 + parts["w_c_rows"] + parts["emb_rows"]
    # fp32 inputs double every stored element
    s32 = shape(dtype="f32")
    t32, b32, p32 = bench.algorithmic_bytes(s32, tokens, parents, depth)
    assert p32["w_c_rows"] == 2 * parts["w_c_rows"] and p32["emb_rows"] == 2 * parts["emb_rows"]
    assert t32 == 2 * 4 * 1000 * 4 + 2 * 4 * 8 * 8


def test_a_chain_expands_every_position_but_the_last():
    s = shape(B=1, n=3, max_depth=3)
    topm, build, parts = bench.algorithmic_bytes(s, np.zeros((1, 3)), np.array([[-1, 0, 1]]), np.array([[1, 2, 3]]))
    assert parts["w_c_rows"] == 3 * 8 * 16 * 2 and parts["emb_rows"] == 2 * 24 * 2


def test_topm_launch_count():
    sms = 152
    assert bench.topm_launches(synth.shape(1), sms) == 1     # 16 rows x 5 chunks: one launch
    assert bench.topm_launches(synth.shape(2), sms) == 2     # 1024 rows: filter, then its selection launch
    assert bench.topm_launches(synth.shape(0), sms) == 1
    # the bound is 6 CTAs per SM: 912 chunks here
    assert bench.topm_launches(shape(B=1, K=912, V=32768), sms) == 1
    assert bench.topm_launches(shape(B=1, K=913, V=32768), sms) == 2
    assert bench.topm_launches(shape(B=1, K=456, V=32768, dtype="f32"), sms) == 1   # fp32 chunks hold 16384
    assert bench.topm_launches(shape(B=1, K=457, V=32768, dtype="f32"), sms) == 2


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6800.0, "fallback")
    assert bench.measured_bf16_tflops() == (1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6667.2}))
    assert bench.measured_peaks() == (6667.2, "measured")
    assert bench.measured_bf16_tflops() == (1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6667.2, "bf16_tflops": 2100}))
    assert bench.measured_bf16_tflops() == (2100.0, "measured")


def test_traffic_counts_only_on_its_own_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("dt_topm", "w") is None                      # no committed figures
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"dt_topm": {"w": {"source_sha": "aaaa", "dram_bytes_per_call": 123}}}))
    monkeypatch.setattr(bench, "source_sha", lambda call: "aaaa")
    assert bench.ncu_traffic("dt_topm", "w") == 123
    assert bench.ncu_traffic("dt_topm", "other") is None                  # another workload
    assert bench.ncu_traffic("dt_build_trees", "w") is None               # another call
    monkeypatch.setattr(bench, "source_sha", lambda call: "bbbb")         # the kernel changed since
    assert bench.ncu_traffic("dt_topm", "w") is None


def test_source_hash_covers_every_listed_file():
    h = bench.source_sha("dt_build_trees")
    assert len(h) == 16 and h != bench.source_sha("dt_topm")
    for files in bench.CALL_SOURCES.values():
        for f in files:
            assert os.path.exists(os.path.join(bench.ROOT, "speculative_decoding_tree_top_gb300", "csrc", f)), f


def test_committed_traffic_is_keyed_by_workload_names():
    # the committed figures are looked up by the workloads' names: they must stay names the bench uses
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    names = {w for call in ("dt_topm", "dt_build_trees") for w in d.get(call, {})}
    assert names and names <= {synth.shape(c).name for c in range(5)}


class FakeNvml:
    """Answers the read-only NVML queries the clock sampler makes: SM clocks from a list, one reasons word."""

    def __init__(self, clocks, reasons, max_mhz=2070, init_rc=0):
        self.clocks, self.reasons, self.max_mhz, self.init_rc, self.i = clocks, reasons, max_mhz, init_rc, 0

    def nvmlInit_v2(self):
        return self.init_rc

    def nvmlDeviceGetHandleByIndex_v2(self, index, ref):
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, kind, ref):
        ref._obj.value = self.max_mhz
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, ref):
        ref._obj.value = self.clocks[self.i % len(self.clocks)]
        self.i += 1
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, ref):
        ref._obj.value = self.reasons
        return 0


def sample(monkeypatch, fake):
    def cdll(name):
        if fake is None:
            raise OSError(name)
        return fake
    monkeypatch.setattr(bench.ctypes, "CDLL", cdll)
    with bench.ClockSampler(0, period_s=0.001) as cs:
        bench.time.sleep(0.05)
    return cs.summary()


def test_clock_sampler_reports_median_clock_and_reasons(monkeypatch):
    s = sample(monkeypatch, FakeNvml([2070, 1950, 2070], 0x4 | 0x1))  # sw_power_cap while busy, idle in between
    assert s["source"] == "nvml" and s["samples"] > 3
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]  # idle is not a throttle
    s = sample(monkeypatch, FakeNvml([1500], 0x8 | 0x40))
    assert s["sm_mhz"] == 1500 and s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_clock_sampler_without_nvml(monkeypatch):
    for fake in (None, FakeNvml([2070], 0, init_rc=1)):  # no library; a library that does not start
        s = sample(monkeypatch, fake)
        assert s["source"] == "unavailable" and s["sm_mhz"] is None and s["samples"] == 0
