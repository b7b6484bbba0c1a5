#!/usr/bin/env python
"""Throughput of one DominoTree drafting round on GB300: dt_topm + dt_build_trees, trees per second.

A step is one whole round over one batch of synthetic inputs already resident in HBM: the top-M of every
(request, position) row over the full vocabulary, then the best-first conditional tree of every request. The default
workload is the Qwen3-4B-shaped single request (B=1, V=151936, K=16, M=64, E=2560, H=512, n=16, T=0).

Timing: W untimed warm-up steps; then K steps, each one dt_round call (dt_topm then dt_build_trees) timed with
CUDA events on the launching stream around the round. The per-call split (and the
builder's roofline) comes from a second pass of the two calls made separately, with events between them. L2 is
flushed between steps outside the events by a 256 MB memset followed by a 256 MB read of another buffer (so the
written lines are not written back inside the next timed call); barrier + synchronize on both sides; max over
ranks. ``e2e`` runs the same rounds through the host-buffer API (pinned logits
and h0 copied in, the tree copied out, every step). The SM clock is sampled through NVML during the timed region.
``graph_replay`` (and ``e2e.graph_replay``) time the same round (the same host round) replayed from its captured
CUDA graph, after the timed loop; the headline stays the direct call.

``configs`` measures every workload (c0-c4) briefly in the same run: µs per round, trees/s, the top-M's and the gather
stage's bandwidth (the builder's own statistics: correction-row bytes gathered over the longest time one CTA spent
gathering them), the round-level roofline (logits read once plus gathered rows, over HBM bandwidth) and, for c0-c2,
the oracle on one thread.

``--impl reference`` times the CPU oracle (fp64, the plain restatement of the method) on the same workload.
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PAGES_MS_PER_ROUND = 2.31   # the pages' CUDA-graph builder, n=16, M=64, Qwen3-4B, RTX 5080 / A6000 (context only)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, help="workload index (1 = the headline single request)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--with-accept", action="store_true",
                    help="also time dt_accept_paths on the round's trees (synthetic target tokens), reported apart")
    ap.add_argument("--with-lmhead", action="store_true",
                    help="also time dt_lmhead_topm (the projection fused with the top-M) against cuBLAS + dt_topm")
    ap.add_argument("--with-attention", action="store_true",
                    help="also time dt_tree_attention (the verify pass over a prefix and the tree) on the workload's batch")
    ap.add_argument("--prefix", type=int, default=2048, help="prefix length of --with-attention")
    ap.add_argument("--builder", choices=["conditional", "marginal"], default="conditional",
                    help="conditional: dt_build_trees (the method); marginal: dt_build_trees_marginal (DDTree scoring)")
    ap.add_argument("--reference-budget", type=float, default=150.0, help="seconds for the whole reference arm")
    ap.add_argument("--configs", default="0,1,2,3,4",
                    help="workloads also measured briefly in the same run (the 'configs' block; empty: none)")
    ap.add_argument("--oracle-1t-budget", type=float, default=8.0,
                    help="seconds of single-threaded oracle work per workload of the configs block (c0-c2)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (a job's time is its slowest replica's), by one all-reduce on `device` (the
    process group's: a GPU for NCCL, the CPU for gloo); x itself when there is one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(config: int, rank: int) -> int:
    """Seed of a replica's synthetic inputs: rank 0 draws the workload's own inputs (those of one GPU), every other
    rank a batch of its own."""
    return 1234 + 100 * config + 7919 * rank


def job_throughput(world: int, trees_per_round: int, rounds: int, seconds: float) -> float:
    """Whole-job trees per second: every replica builds `trees_per_round` trees per round (weak scaling), and the job
    takes as long as its slowest replica (`seconds`, already the maximum over ranks)."""
    return world * trees_per_round * rounds / seconds


# ---------------------------------------------------------------------------------------------------------------
class ClockSampler:
    """SM clock and throttle reasons of one GPU, sampled by NVML in a thread (read-only queries)."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value & ~0x1
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": "unavailable"}
        s = sorted(self.samples)
        return {"sm_mhz": s[len(s) // 2], "sm_max_mhz": self.max_mhz,
                "reasons": [v for k, v in self.REASONS.items() if self.reasons & k], "samples": len(s),
                "source": "nvml"}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), "measured"
    return 6800.0, "fallback"


def measured_bf16_tflops():
    """Dense bf16 tensor peak in TFLOP/s for a kernel timed alone (the burst figure), and where it comes from."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("bf16_tflops"):
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# The sources each C-ABI call is built from: a committed ncu figure counts only while they are unchanged.
CALL_SOURCES = {
    "dt_topm": ["topm.cu", "topm_filter.cuh", "topm_select.cuh", "dt_internal.cuh"],
    "dt_build_trees": ["build_trees.cu", "build_small.cu", "build_common.cuh", "umma.cuh", "dt_internal.cuh"],
}


def source_sha(call: str) -> str:
    h = hashlib.sha256()
    for name in CALL_SOURCES[call]:
        with open(os.path.join(ROOT, "speculative_decoding_tree_top_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(call: str, workload: str):
    """DRAM bytes per call from a committed ncu summary, if it was taken on the current sources of the call."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(call, {}).get(workload)
    if not e or e.get("source_sha") != source_sha(call):
        return None
    return e.get("dram_bytes_per_call")


# ---------------------------------------------------------------------------------------------------------------
def topm_launches(shape, sms: int) -> int:
    """Kernels one dt_topm call launches: the filter, plus a selection launch unless the grid is about two waves or
    fewer (then the filter's last CTA of each row selects)."""
    chunk = 16384 if shape.dtype == "f32" else 32768
    chunks = -(-shape.V // chunk)
    return 1 if shape.B * shape.K * chunks <= 6 * sms else 2


def algorithmic_bytes(shape, tokens, parents, depth):
    """Bytes a launch must move at least once (HBM roofline numerators), from the trees actually built.

    dt_topm: the logits once + the ids/values written.
    dt_build_trees: per request, the W_c rows of every block position it expanded (M rows of H per position; nodes of
    the same depth share them), one embedding row per GRU step, the GRU weights once (shared by the batch), the
    top-M ids/values and h0 read, the tree written."""
    s = 4 if shape.dtype == "f32" else 2
    B, K, V, M, H, E, n = shape.B, shape.K, shape.V, shape.M, shape.H, shape.E, shape.n
    topm = B * K * V * s + B * K * M * 8
    wc = emb = 0
    for b in range(B):
        expanded = {0}   # the root expands into position 0
        gru = 0
        for i in range(n - 1):
            if depth[b, i] < shape.max_depth:
                expanded.add(int(depth[b, i]))
                gru += 1
        wc += len(expanded) * M * H * s
        emb += gru * E * s
    gru_w = 3 * H * (E + H) * s + 6 * H * s
    build = wc + emb + gru_w + B * K * M * 8 + B * H * 4 + B * n * 16 + B * n * n
    return topm, build, dict(w_c_rows=wc, emb_rows=emb, gru_weights=gru_w)


def round_bytes(shape, parts):
    """The round-level roofline numerator: the logits read once plus the gathered rows (W_c rows of the expanded
    block positions and the expansions' embedding rows), from the trees actually built."""
    s = 4 if shape.dtype == "f32" else 2
    return shape.B * shape.K * shape.V * s + parts["w_c_rows"] + parts["emb_rows"]


def oracle_single_thread(inp, budget_s):
    """The oracle on one thread: whole rounds of a bounded sample of the workload's requests, for about budget_s."""
    import numpy as np
    from oracle import oracle as orc
    from speculative_decoding_tree_top_gb300.synth import host_array
    s = inp.shape
    logits = host_array(inp.logits)
    h0 = host_array(inp.h0).astype(np.float64)
    w = orc.weights_of(inp)
    trees, t0 = 0, time.perf_counter()
    b = 0
    while True:
        ids, vals = orc.topm(np.ascontiguousarray(logits[b:b + 1]), s.M, threads=1)
        orc.build_trees(ids, vals, h0[b:b + 1], w, s.n, s.max_depth, s.T, threads=1)
        trees += 1
        b = (b + 1) % s.B
        el = time.perf_counter() - t0
        if el >= budget_s or (trees >= s.B and el >= 0.25 * budget_s):
            break
    return {"trees_per_sec": round(trees / el, 3), "s_per_tree": round(el / trees, 4), "cores": 1,
            "sample": f"{trees} whole trees (top-M of the request's {s.K} rows, then its tree) in {el:.1f} s"}


def measure_configs(args, dev, flush_l2, stream, peak):
    """Every workload briefly, in the same process: round time, the per-call split, the stages' bandwidth, the
    round-level roofline, and (c0-c2) the oracle on one thread."""
    import numpy as np
    import torch
    from speculative_decoding_tree_top_gb300 import dominotree as dt, synth
    out = {}
    steps_of = {0: 50, 1: 50, 2: 30, 3: 30, 4: 15}
    for c in [int(x) for x in args.configs.split(",") if x.strip() != ""]:
        s = synth.shape(c)
        inp = synth.make_inputs(c, device=dev, seed=1234 + 100 * c)
        w = dt.Weights.of(inp)
        rnd = dt.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w, device=dev)
        for _ in range(3):
            rnd.round(inp.logits, inp.h0, stream)
        steps = steps_of.get(c, 20)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        torch.cuda.synchronize()
        for e in ev:
            flush_l2()
            e[0].record(stream)
            rnd.round(inp.logits, inp.h0, stream)
            e[1].record(stream)
            flush_l2()
            e[2].record(stream)
            rnd.topm(inp.logits, stream)
            e[3].record(stream)
            rnd.build(inp.h0, stream)
            e[4].record(stream)
        torch.cuda.synchronize()
        rnd.check()
        stats = dt.dt_build_stats_read(rnd.workspace, stream)
        r_us = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]) * 1e3)
        t_us = float(np.mean([e[2].elapsed_time(e[3]) for e in ev]) * 1e3)
        b_us = float(np.mean([e[3].elapsed_time(e[4]) for e in ev]) * 1e3)
        o = {k: v.cpu().numpy() for k, v in rnd.out.items()}
        topm_b, build_b, parts = algorithmic_bytes(s, o["tokens"], o["parents"], o["depth"])
        rb = round_bytes(s, parts)
        gather_gbps = stats["gather_bytes"] / stats["gather_ns"] if stats["gather_ns"] else None
        d = {"workload": s.describe(), "steps": steps, "us_per_round": round(r_us, 2),
             "trees_per_sec": round(s.B / (r_us * 1e-6), 1),
             "dt_topm": {"us": round(t_us, 2), "gbps": round(topm_b / (t_us * 1e3), 1),
                         "frac_of_hbm_peak": round(topm_b / (t_us * 1e3) / peak, 4)},
             "dt_build_trees": {"us": round(b_us, 2), "waves": stats["waves"], "expansions": stats["expansions"],
                                "gather": {"bytes": stats["gather_bytes"], "ns": stats["gather_ns"],
                                           "gbps": round(gather_gbps, 1) if gather_gbps else None,
                                           "frac_of_hbm_peak": round(gather_gbps / peak, 4) if gather_gbps else None}},
             "round_roofline": {"bytes": rb, "us_at_peak": round(rb / (peak * 1e3), 3),
                                "frac": round(rb / (r_us * 1e3) / peak, 4)}}
        if c <= 2 and args.oracle_1t_budget > 0:
            d["oracle_1_thread"] = oracle_single_thread(inp, args.oracle_1t_budget)
        out[f"c{c}"] = d
        del rnd, inp, w
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    import numpy as np
    import torch
    from speculative_decoding_tree_top_gb300 import dominotree as dt, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    s = synth.shape(args.config)
    inp = synth.make_inputs(args.config, device=dev, seed=replica_seed(args.config, rank))
    w = dt.Weights.of(inp)
    rnd = dt.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w, device=dev)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        # Write a buffer twice the size of L2, then read another one: nothing of the step's inputs stays cached,
        # and the written lines are written back here rather than inside the next timed call.
        flush_w.zero_()
        flush_r.max()

    stream = torch.cuda.current_stream()
    marginal = args.builder == "marginal"

    def step(evs=None):
        flush_l2()
        if evs:
            evs[0].record(stream)
        rnd.topm(inp.logits, stream)
        if evs:
            evs[1].record(stream)
        if marginal:
            rnd.build_marginal(stream)
        else:
            rnd.build(inp.h0, stream)
        if evs:
            evs[2].record(stream)

    def step_round(evs):
        # the headline: one dt_round call, events around the round only
        flush_l2()
        evs[0].record(stream)
        rnd.round(inp.logits, inp.h0, stream)
        evs[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rnd.check()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if not marginal:
        for _ in range(args.warmup):
            step_round([torch.cuda.Event(enable_timing=True) for _ in range(2)])
    barrier()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            (step if marginal else step_round)(evs[i])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier()
    rnd.check()
    if marginal:
        topm_ms = np.array([a.elapsed_time(b) for a, b, _ in evs])
        build_ms = np.array([b.elapsed_time(c) for _, b, c in evs])
        round_ms = topm_ms + build_ms
    else:
        round_ms = np.array([a.elapsed_time(b) for a, b, _ in evs])
        # the per-call split (and the builder's roofline): the two calls made one after the other, events between
        split_steps = min(args.steps, 100)
        sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(split_steps)]
        for i in range(split_steps):
            step(sevs[i])
        torch.cuda.synchronize()
        rnd.check()
        topm_ms = np.array([a.elapsed_time(b) for a, b, _ in sevs])
        build_ms = np.array([b.elapsed_time(c) for _, b, c in sevs])
        # the same round replayed from its captured CUDA graph (Round.capture): the same two launches without their
        # host-side work, L2 flushed before each replay like the headline's rounds
        graph = rnd.capture(inp.logits, inp.h0)
        gevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(split_steps)]
        for a, b in gevs:
            flush_l2()
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        rnd.check()
        graph_ms = np.array([a.elapsed_time(b) for a, b in gevs])
        del graph
    total_s = max_over_ranks(float(round_ms.sum()) / 1e3, world, dev)
    value = job_throughput(world, s.B, args.steps, total_s)

    out = {k: v.cpu().numpy() for k, v in rnd.out.items()}
    topm_b, build_b, parts = algorithmic_bytes(s, out["tokens"], out["parents"], out["depth"])
    if marginal:  # no GRU, no correction rows: the candidates' ids and values read, the tree written
        build_b = s.B * s.K * s.M * 8 + s.B * s.n * 16 + s.B * s.n * s.n
        parts = dict(ids_vals=s.B * s.K * s.M * 8)
    peak, peak_src = measured_peaks()
    kernels = {
        "dt_topm": dict(us=float(topm_ms.mean() * 1e3), bytes=topm_b, gbps=topm_b / (topm_ms.mean() * 1e6),
                        sources=CALL_SOURCES["dt_topm"]),
        "dt_build_trees": dict(us=float(build_ms.mean() * 1e3), bytes=build_b,
                               gbps=build_b / (build_ms.mean() * 1e6), sources=CALL_SOURCES["dt_build_trees"]),
    }
    dom = max(kernels, key=lambda k: kernels[k]["us"])
    kd = kernels[dom]
    traffic = ncu_traffic(dom, s.name)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(kd["gbps"], 1), "peak": peak, "unit": "GB/s",
                "frac": round(kd["gbps"] / peak, 4), "traffic": traffic, "peak_source": peak_src,
                "algorithmic_bytes_per_launch": kd["bytes"], "bytes_breakdown": parts if dom == "dt_build_trees"
                else {"logits": s.B * s.K * s.V * (4 if s.dtype == "f32" else 2)}}

    if args.with_accept:  # the step after verification, timed on its own (inputs resident, after the timed loop)
        tn = torch.from_numpy(synth.make_target_next(out["tokens"], out["parents"], s.V, 0.9, seed=rank)).to(dev)
        acc_out = dt.dt_accept_paths(rnd.out["tokens"], rnd.out["parents"], tn, stream=stream)
        for _ in range(args.warmup):
            dt.dt_accept_paths(rnd.out["tokens"], rnd.out["parents"], tn, acc_out, stream)
        # a launch of one warp per request is shorter than its host-side call, so the calls are captured in a CUDA
        # graph and replayed: the events then time the GPU, not the Python caller
        reps = 32
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side), torch.cuda.graph(graph, stream=side):
            for _ in range(reps):
                dt.dt_accept_paths(rnd.out["tokens"], rnd.out["parents"], tn, acc_out, side)
        stream.wait_stream(side)
        graph.replay()
        ea = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        torch.cuda.synchronize()
        for a, b in ea:
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        acc_ms = np.array([a.elapsed_time(b) for a, b in ea]) / reps
        kernels["dt_accept_paths"] = dict(us=float(acc_ms.mean() * 1e3), bytes=s.B * s.n * 8 + s.B * (s.n + 1) * 4,
                                          mean_accept_len=float(acc_out["accept_len"].float().mean().item()),
                                          sources=["accept.cu"])

    if args.with_lmhead and s.dtype == "bf16":
        # The drafter's projection of the R = B*K backbone hidden states (width E) onto the vocabulary, fused with
        # its top-M, against the unfused path: the cuBLAS GEMM writes the logits, dt_topm reads them back.
        R = s.B * s.K
        hid, head = (t.to(dev) for t in synth.make_lmhead_inputs(R, s.E, s.V, seed=777 + rank))
        lws = dt.new_workspace(dt.dt_lmhead_workspace_bytes(R, s.E, s.V, s.M), dev)
        l_ids = torch.empty((R, s.M), dtype=torch.int32, device=dev)
        l_vals = torch.empty((R, s.M), dtype=torch.float32, device=dev)
        u_logits = torch.empty((1, R, s.V), dtype=torch.bfloat16, device=dev)
        u_ids = torch.empty((1, R, s.M), dtype=torch.int32, device=dev)
        u_vals = torch.empty((1, R, s.M), dtype=torch.float32, device=dev)
        tws = dt.new_workspace(dt.dt_topm_workspace_bytes(1, R, s.V, s.M), dev)

        def fused():
            dt.dt_lmhead_topm(hid, head, s.M, l_ids, l_vals, lws, stream)

        def unfused(ev=None):
            torch.matmul(hid, head.t(), out=u_logits[0])
            if ev is not None:
                ev.record(stream)
            dt.dt_topm(u_logits, s.M, u_ids, u_vals, tws, stream)

        for _ in range(args.warmup):
            fused()
            unfused()
        steps = max(20, min(args.steps, 200))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        torch.cuda.synchronize()
        for e in ev:
            flush_l2()
            e[0].record(stream)
            fused()
            e[1].record(stream)
            flush_l2()
            e[2].record(stream)
            unfused(e[3])
            e[4].record(stream)
        torch.cuda.synchronize()
        f_us = np.array([e[0].elapsed_time(e[1]) for e in ev]) * 1e3
        g_us = np.array([e[2].elapsed_time(e[3]) for e in ev]) * 1e3
        t_us = np.array([e[3].elapsed_time(e[4]) for e in ev]) * 1e3
        lbytes = s.V * s.E * 2 + R * s.E * 2 + R * s.M * 8
        bf16_peak, _ = measured_bf16_tflops()
        # the unfused logits are rounded to bf16 by the GEMM, the fused ones stay fp32: near-ties may differ
        a, b = l_ids.cpu().numpy(), u_ids[0].cpu().numpy()
        common = float(np.mean([len(set(a[r]) & set(b[r])) / s.M for r in range(R)]))
        kernels["dt_lmhead_topm"] = dict(
            us=float(f_us.mean()), bytes=lbytes, gbps=lbytes / (f_us.mean() * 1e3),
            frac_of_hbm_peak=round(lbytes / (f_us.mean() * 1e3) / peak, 4),
            tflops=2.0 * R * s.E * s.V / (f_us.mean() * 1e6),
            frac_of_bf16_peak=round(2.0 * R * s.E * s.V / (f_us.mean() * 1e6) / bf16_peak, 4), rows=R, width=s.E,
            path="one launch, logits in tensor memory" if R <= 64 else "blocked passes (pool, bound, filter, select)",
            unfused_us=dict(cublas_projection=float(g_us.mean()), dt_topm=float(t_us.mean()),
                            total=float((g_us + t_us).mean())),
            ids_shared_with_unfused=round(common, 4), sources=["lmhead_topm.cu", "topm_select.cuh", "umma.cuh"])

    if args.with_attention:
        # The target's verify pass over the accepted prefix and the n tree nodes, Qwen3-4B's attention shape (32
        # query heads over 8 key/value heads, d = 128), with the ancestor masks of this step's own trees; against
        # torch's scaled_dot_product_attention with the same boolean mask (context).
        Hq, Hkv, d, Lp = 32, 8, 128, args.prefix
        aq, ak, av, _ = (t.to(dev) for t in synth.make_attention_inputs(s.B, s.n, Lp, Hq, Hkv, d, seed=99 + rank))
        amask = rnd.out["mask"]
        aws = dt.new_workspace(dt.dt_tree_attention_workspace_bytes(s.B, s.n, Lp, Hq, Hkv, d), dev)
        aout = torch.empty((s.B, s.n, Hq, d), dtype=torch.float32, device=dev)
        scale = 1.0 / math.sqrt(d)
        bm = torch.ones((s.B, 1, s.n, Lp + s.n), dtype=torch.bool, device=dev)
        bm[:, 0, :, Lp:] = amask.bool()
        qt = aq.permute(0, 2, 1, 3)

        def sdpa():
            return torch.nn.functional.scaled_dot_product_attention(qt, ak, av, attn_mask=bm, scale=scale,
                                                                    enable_gqa=True)

        for _ in range(args.warmup):
            dt.dt_tree_attention(aq, ak, av, amask, scale, aout, aws, stream)
            sdpa()
        steps = max(20, min(args.steps, 200))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        torch.cuda.synchronize()
        for e in ev:
            flush_l2()
            e[0].record(stream)
            dt.dt_tree_attention(aq, ak, av, amask, scale, aout, aws, stream)
            e[1].record(stream)
            flush_l2()
            e[2].record(stream)
            sdpa()
            e[3].record(stream)
        torch.cuda.synchronize()
        a_us = np.array([e[0].elapsed_time(e[1]) for e in ev]) * 1e3
        s_us = np.array([e[2].elapsed_time(e[3]) for e in ev]) * 1e3
        abytes = 2 * s.B * Hkv * (Lp + s.n) * d * 2 + s.B * s.n * Hq * d * (2 + 4) + s.B * s.n * s.n
        diff = float((sdpa().permute(0, 2, 1, 3).float() - aout).abs().max().item())
        kernels["dt_tree_attention"] = dict(
            us=float(a_us.mean()), bytes=abytes, gbps=abytes / (a_us.mean() * 1e3),
            frac_of_hbm_peak=round(abytes / (a_us.mean() * 1e3) / peak, 4), prefix=Lp, heads=[Hq, Hkv, d],
            torch_sdpa_us=float(s_us.mean()), max_abs_diff_vs_sdpa=round(diff, 5),
            sources=["tree_attn.cu"])

    e2e = None
    if not args.no_e2e and not marginal:
        hr = dt.HostRound(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w, inp.logits.dtype, device=dev)
        hr.host_logits.copy_(inp.logits)  # the step's inputs, in the round's pinned input buffer
        hr.host_h0.copy_(inp.h0)
        for _ in range(args.warmup):
            hr.run()
        torch.cuda.synchronize()
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier()
        for i in range(args.steps):
            flush_l2()
            ev2[i][0].record(stream)
            hr.run()
            ev2[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        hr.check()
        assert np.array_equal(hr.host_out["tokens"].numpy(), out["tokens"]), "host-buffer round differs"
        e2e_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev2) / 1e3, world, dev)
        e2e = {"value": round(job_throughput(world, s.B, args.steps, e2e_s), 2), "unit": "trees/s",
               "h2d_bytes_per_step": hr.h2d_bytes(), "d2h_bytes_per_step": hr.d2h_bytes(),
               "us_per_round": round(e2e_s / args.steps * 1e6, 2)}
        # the same host rounds replayed from their captured CUDA graph (HostRound.capture: the copy in, the round's
        # launches and the copy out as graph nodes), up to 100 of them, L2 flushed before each
        hgraph = hr.capture()
        hevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(min(args.steps, 100))]
        for a, b in hevs:
            flush_l2()
            a.record(stream)
            hgraph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        hr.check()
        assert np.array_equal(hr.host_out["tokens"].numpy(), out["tokens"]), "replayed host round differs"
        hg_us = float(np.mean([a.elapsed_time(b) for a, b in hevs])) * 1e3
        e2e["graph_replay"] = {"us_per_round": round(hg_us, 2), "trees_per_s": round(world * s.B / (hg_us / 1e6), 2),
                               "rounds": len(hevs)}
        del hgraph

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not marginal:
        cpu = cpu_baseline(inp, args.cpu_budget)

    rbytes = round_bytes(s, parts) if not marginal else None
    round_roofline = None if marginal else {
        "bytes": rbytes, "achieved_gbps": round(rbytes / (total_s / args.steps * 1e9), 1), "peak": peak,
        "frac": round(rbytes / (total_s / args.steps * 1e9) / peak, 4),
        "definition": "logits read once plus the gathered W_c and embedding rows, over HBM bandwidth, per round"}
    configs = None
    if rank == 0 and world == 1 and not marginal and args.configs.strip():
        configs = measure_configs(args, dev, flush_l2, stream, peak)

    if rank != 0:
        return None
    return {
        "metric": "trees_per_sec", "value": round(value, 2), "unit": "trees/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_s / args.steps * 1e3, 5),
        "us_per_round": round(total_s / args.steps * 1e6, 2),
        "us_per_round_two_calls": round(float((topm_ms + build_ms).mean()) * 1e3, 2),
        "graph_replay": None if marginal else {
            "us_per_round": round(float(graph_ms.mean()) * 1e3, 2),
            "trees_per_s": round(world * s.B / (float(graph_ms.mean()) / 1e3), 2), "rounds": int(graph_ms.size)},
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(value / (1e3 / PAGES_MS_PER_ROUND), 3) if args.config == 1 else None,
        "dtype": "f32", "inputs_dtype": s.dtype, "data": "synthetic",
        "config": {"workload": s.describe() + (" marginal-scoring" if marginal else ""), "B_per_gpu": s.B,
                   "l2": "flushed between steps outside the timed events: a 256 MB memset, then a 256 MB read of another buffer"},
        "kernels": {k: {kk: (round(vv, 3) if isinstance(vv, float) else vv) for kk, vv in d.items()}
                    for k, d in kernels.items()},
        "roofline": roofline, "round_roofline": round_roofline, "configs": configs, "e2e": e2e,
        "cpu_baseline": cpu, "gpu_launches": (topm_launches(s, torch.cuda.get_device_properties(dev).multi_processor_count) + 1) * args.steps,
        "clocks": clocks.summary(), "wall_s_timed_loop": round(t_wall, 4),
    }


def cpu_baseline(inp, budget_s):
    """The oracle as it stands, on whole rounds of the same workload, for about ``budget_s`` seconds."""
    import numpy as np
    from oracle import oracle as orc
    from speculative_decoding_tree_top_gb300.synth import host_array
    s = inp.shape
    logits = host_array(inp.logits)
    h0 = host_array(inp.h0).astype(np.float64)
    w = orc.weights_of(inp)
    threads = len(os.sched_getaffinity(0))
    rounds, t0 = 0, time.perf_counter()
    while True:
        ids, vals = orc.topm(logits, s.M, threads=threads)
        orc.build_trees(ids, vals, h0, w, s.n, s.max_depth, s.T, threads=threads)
        rounds += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(rounds * s.B / el, 3), "unit": "trees/s", "cores": threads, "kind": "oracle",
            "sample": f"{rounds} whole rounds of {s.name} (B={s.B}) in {el:.1f} s, OpenMP over rows and requests"}


def run_reference(args, world, rank):
    """The CPU oracle timed as the reference arm, on the same workload, metric and unit."""
    import numpy as np
    import torch
    from oracle import oracle as orc
    from speculative_decoding_tree_top_gb300 import synth
    from speculative_decoding_tree_top_gb300.synth import host_array
    if rank != 0:
        return None
    s = synth.shape(args.config)
    inp = synth.make_inputs(args.config, device="cuda" if torch.cuda.is_available() else "cpu")
    logits = host_array(inp.logits)
    h0 = host_array(inp.h0).astype(np.float64)
    w = orc.weights_of(inp)
    threads = len(os.sched_getaffinity(0))

    def one(frac):
        # a bounded sample of one round: the top-M of a share of the rows and the tree with a share of the pops
        rows = max(1, math.ceil(s.K * frac))
        n = max(1, math.ceil(s.n * frac))
        ids, vals = orc.topm(np.ascontiguousarray(logits[:, :rows]), s.M, threads=threads)
        if rows < s.K:
            full_ids = np.zeros((s.B, s.K, s.M), np.int32)
            full_vals = np.zeros((s.B, s.K, s.M), np.float64)
            full_ids[:, :rows], full_vals[:, :rows] = ids, vals
            full_ids[:, rows:], full_vals[:, rows:] = ids[:, -1:], vals[:, -1:]
            ids, vals = full_ids, full_vals
        orc.build_trees(ids, vals, h0, w, n, s.max_depth, s.T, threads=threads)
        return min(rows / s.K, n / s.n)

    t0 = time.perf_counter()
    one(1.0)
    est = time.perf_counter() - t0
    frac = min(1.0, args.reference_budget / max(1e-9, (args.steps + args.warmup) * est))
    for _ in range(max(0, args.warmup - 1)):
        one(frac)
    t0 = time.perf_counter()
    done = 0.0
    for _ in range(args.steps):
        done += one(frac)
    el = time.perf_counter() - t0
    value = done * s.B / el
    sample = (f"each step: one whole round of {s.name}" if frac >= 1.0 else
              f"each step: top-M of {max(1, math.ceil(s.K * frac))}/{s.K} rows and {max(1, math.ceil(s.n * frac))}"
              f"/{s.n} pops of one round, counted as that share of a tree")
    return {"impl": "reference", "metric": "trees_per_sec", "value": round(value, 3), "unit": "trees/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": s.describe(), "B_per_gpu": s.B},
            "cpu_baseline": {"value": round(value, 3), "unit": "trees/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "trees/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
