"""dt_build_trees on the GPU against the CPU oracle: structure bit-exact up to the first near-tie (gap <= 1e-3),
scores within 1e-3 of the oracle's fp64 rescoring of the GPU's own tree, tree invariants everywhere."""
import zlib

import numpy as np
import pytest
import torch

from oracle import compare
from speculative_decoding_tree_top_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 1e-3


# The stricter pass: two pops count as a near-tie only when the oracle's gap is <= 5e-5, eight times the largest
# fp32-vs-fp64 score difference seen on these workloads (6e-6); beyond that the builders must decide alike.
STRICT = 5e-5


def run_both(dtlib, orc, inp):
    s = inp.shape
    w = dtlib.Weights.of(inp)
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w, device="cuda")
    out = rnd(inp.logits, inp.h0)
    torch.cuda.synchronize()
    rnd.check()
    ora = orc.round_(inp)
    assert np.array_equal(rnd.ids.cpu().numpy(), ora["ids"])
    gpu = {k: v.cpu().numpy() for k, v in out.items()}
    h0 = synth.host_array(inp.h0).astype(np.float64)
    resc = orc.rescore(ora["ids"], ora["vals"], h0, orc.weights_of(inp), gpu["tokens"], gpu["parents"],
                       gpu["depth"], s.max_depth, s.T)
    rep = compare.compare_round(gpu, ora, resc, s.n, s.max_depth, TOL)
    strict = compare.compare_round(gpu, ora, resc, s.n, s.max_depth, TOL, struct_tol=STRICT)
    rep["compared_pops_strict"] = strict["compared_pops"]
    return rep, gpu, ora, rnd


@pytest.mark.parametrize("config", [0, 1, 2, 3, 4])
def test_build_parity_workloads(dtlib, orc, config):
    inp = synth.make_inputs(config, device="cuda")
    rep, *_ = run_both(dtlib, orc, inp)
    print(config, rep)
    # not vacuous: under the stricter pass most pops are compared bit-exactly (the rest follow a genuine
    # near-tie of the oracle, where either choice is correct), and past the first near-tie every node clear of the
    # n-th score is in both trees (on these workloads the node-set check covers all but the nodes at the boundary,
    # 0.875-0.98 of them)
    assert rep["compared_pops"] >= 0.5 and rep["compared_pops_strict"] >= 0.8 and rep["top_nodes"] >= 0.5


def tiny(seed, **kw):
    base = dict(B=2, V=600, K=5, M=6, H=16, E=24, n=12, max_depth=4, T=0.0, dtype="f32", logit_scale=3.0,
                boost_count=8, boost_lo=2.0, boost_hi=6.0, name="edge")
    base.update(kw)
    return synth.make_inputs(synth.Shape(**base), device="cuda", seed=seed)


@pytest.mark.parametrize("kw", [
    dict(M=1, n=4, max_depth=4),                         # a chain, all scores 0
    dict(max_depth=1, n=5),                              # the best children of the root
    dict(n=1),                                           # the arg-max
    dict(M=2, n=30, max_depth=4, K=4),                   # the whole depth-limited tree (2+4+8+16)
    dict(B=300, n=10),                                   # more requests than SMs
    dict(H=24, E=40, n=20, T=0.5),                       # widths that are not multiples of the tile
    dict(dtype="bf16", n=25, T=2.0),
    dict(dtype="bf16", M=40, n=64, max_depth=5, K=5),    # a wide, deep frontier
    dict(B=3, V=9000, M=100, n=40, T=1.0, logit_scale=0.5),
    dict(dtype="bf16", B=20, E=64, H=64, n=20),          # tensor-core GRU with fewer K blocks than K splits
    dict(dtype="bf16", B=153, E=128, H=64, M=16, n=20),  # tensor-core GRU, one CTA owning two requests (a batched
                                                         # control phase and its staged activation rows)
])
def test_build_edge_cases(dtlib, orc, kw):
    inp = tiny(zlib.crc32(str(sorted(kw.items())).encode()) % 10000, **kw)  # a seed fixed by the case
    run_both(dtlib, orc, inp)


def test_build_without_biases(dtlib, orc):
    s = synth.Shape(B=2, V=600, K=4, M=5, H=16, E=16, n=15, max_depth=4, T=0.0, dtype="bf16", name="nobias")
    inp = synth.make_inputs(s, device="cuda", seed=5, biases=False)
    run_both(dtlib, orc, inp)


def test_build_deterministic(dtlib, orc):
    inp = synth.make_inputs(2, device="cuda")
    s = inp.shape
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, dtlib.Weights.of(inp))
    a = {k: v.clone() for k, v in rnd(inp.logits, inp.h0).items()}
    b = rnd(inp.logits, inp.h0)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_barrier_timeout_is_reported_and_recoverable(dtlib, orc):
    """With a zero wait budget the first barrier wait gives up at once: the kernel records DT_ERR_TIMEOUT and
    returns (no hang, no fault); after re-initialising the workspace the next round is correct."""
    inp = synth.make_inputs(0, device="cuda")
    s = inp.shape
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, dtlib.Weights.of(inp))
    try:
        dtlib.dt_set_barrier_timeout_ns(0)
        rnd(inp.logits, inp.h0)
        assert dtlib.dt_get_error(rnd.workspace) == dtlib.Status.TIMEOUT
    finally:
        dtlib.dt_set_barrier_timeout_ns(2_000_000_000)
    dtlib.dt_workspace_init(rnd.workspace)
    out = rnd(inp.logits, inp.h0)
    torch.cuda.synchronize()
    rnd.check()
    ora = orc.round_(inp)
    assert np.array_equal(out["tokens"].cpu().numpy(), ora["tokens"])


def test_rounds_reuse_one_workspace(dtlib, orc):
    """Consecutive rounds on one workspace (top-M region then the builder's region): no state leaks between calls."""
    s = synth.shape(2, B=8)
    inputs = [synth.make_inputs(s, device="cuda", seed=seed) for seed in (1, 2)]
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, dtlib.Weights.of(inputs[0]))
    expect = [orc.round_(inp) for inp in inputs]
    for i in (0, 1, 0, 1, 1, 0):
        inp = inputs[i]
        rnd.weights = dtlib.Weights.of(inp)
        out = rnd(inp.logits, inp.h0)
        torch.cuda.synchronize()
        rnd.check()
        assert np.array_equal(rnd.ids.cpu().numpy(), expect[i]["ids"])
        gpu = {k: v.cpu().numpy() for k, v in out.items()}
        h0 = synth.host_array(inp.h0).astype(np.float64)
        resc = orc.rescore(expect[i]["ids"], expect[i]["vals"], h0, orc.weights_of(inp), gpu["tokens"],
                           gpu["parents"], gpu["depth"], s.max_depth, s.T)
        compare.compare_round(gpu, expect[i], resc, s.n, s.max_depth, TOL, struct_tol=STRICT)


def test_out_of_range_ids_are_reported_not_gathered(dtlib):
    """Candidate ids are caller input: one outside [0, V) must come back as a device status, never as a gather
    outside the weight arrays (the kernel range-checks every id before using it)."""
    inp = synth.make_inputs(0, device="cuda")
    s = inp.shape
    ids, vals = dtlib.dt_topm(inp.logits, s.M)
    ids[0, 0, 3] = s.V + 1000
    ids[0, 1, 0] = -7
    ws = dtlib.new_workspace(dtlib.dt_build_workspace_bytes(s.B, s.K, s.V, s.M, s.n, s.H, s.E))
    out = dtlib.dt_build_trees(ids, vals, inp.h0, dtlib.Weights.of(inp), s.n, s.max_depth, s.T, workspace=ws)
    assert dtlib.dt_get_error(ws) == dtlib.Status.INVALID_ARG
    tok = out["tokens"].cpu().numpy()
    assert tok.min() >= 0 and tok.max() < s.V


@pytest.mark.parametrize("case", [
    dict(config=1),                                                    # one request, the bench workload
    dict(config=0),                                                    # tiny, fp32
    dict(config=2, B=2),                                               # two requests share a wave
    dict(config=3, B=2),                                               # deeper trees (T = 0.5)
    dict(tiny=dict(dtype="bf16", M=40, n=64, max_depth=5, K=5, B=1)),  # wide and deep
    dict(tiny=dict(M=1, n=4, max_depth=4, B=1)),                       # a chain: nothing to look ahead at
    dict(config=2, B=16),                                              # the large-batch builder
    dict(config=3, B=12),                                              # ... deeper trees, H = 1024
    dict(config=4, B=12),                                              # ... M = 128, n = 64
    dict(config=2, B=160),                                             # ... GRU tiles on one CTA each at k = 8,
                                                                       #     K split over CTAs at k = 1
    dict(tiny=dict(B=20, M=6, n=30, max_depth=4)),                     # ... fp32, CUDA-core GRU tiles
])
def test_lookahead_width_does_not_change_the_tree(dtlib, case):
    """Expanding several frontier nodes per wave only changes when children become known, never the pop order:
    every lookahead width gives bit-identical outputs."""
    if "tiny" in case:
        inp = tiny(11, **case["tiny"])
    else:
        inp = synth.make_inputs(synth.shape(case["config"], **{k: v for k, v in case.items() if k != "config"}),
                                device="cuda")
    s = inp.shape
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, dtlib.Weights.of(inp))
    outs = []
    try:
        for k in (1, 2, 3, 8, 0):
            dtlib.dt_set_lookahead(k)
            out = rnd(inp.logits, inp.h0)
            torch.cuda.synchronize()
            rnd.check()
            outs.append({key: v.clone() for key, v in out.items()})
    finally:
        dtlib.dt_set_lookahead(0)
    for o in outs[1:]:
        for key in o:
            assert torch.equal(o[key], outs[0][key]), key


@pytest.mark.parametrize("case", [
    dict(config=1),           # one request
    dict(config=0),           # tiny, fp32
    dict(config=2, B=8),      # the largest small-batch round
    dict(config=2, B=16),     # the large-batch builder: two ordinary launches
])
def test_round_matches_the_two_calls(dtlib, case):
    """dt_round gives bit-identical ids, values and trees to dt_topm followed by dt_build_trees, also with several
    rounds queued back to back on one workspace and no synchronisation between them."""
    s = synth.shape(case["config"], **{k: v for k, v in case.items() if k != "config"})
    inputs = [synth.make_inputs(s, device="cuda", seed=40 + i) for i in range(3)]
    w = dtlib.Weights.of(inputs[0])
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w)
    ref = []
    for inp in inputs:
        rnd.topm(inp.logits)
        out = rnd.build(inp.h0)
        torch.cuda.synchronize()
        rnd.check()
        ref.append(({k: v.clone() for k, v in out.items()}, rnd.ids.clone(), rnd.vals.clone()))
    got = []
    for inp in inputs:  # queued back to back: no synchronisation between the rounds
        out = rnd.round(inp.logits, inp.h0)
        got.append(({k: v.clone() for k, v in out.items()}, rnd.ids.clone(), rnd.vals.clone()))
    torch.cuda.synchronize()
    rnd.check()
    for (ro, ri, rv), (go, gi, gv) in zip(ref, got):
        assert torch.equal(ri, gi) and torch.equal(rv, gv)
        for k in ro:
            assert torch.equal(ro[k], go[k]), k
    # the functional form, with its own buffers, agrees too
    inp = inputs[-1]
    out = dtlib.dt_round(inp.logits, inp.h0, w, s.M, s.n, s.max_depth, s.T)
    torch.cuda.synchronize()
    for k in ref[-1][0]:
        assert torch.equal(ref[-1][0][k], out[k]), k


@pytest.mark.parametrize("case", [dict(config=1), dict(config=2, B=16)])
def test_captured_round_replays_new_inputs(dtlib, case):
    """Round.capture: the CUDA graph of one dt_round call (the top-M and the cooperative builder as graph nodes),
    replayed after each round's inputs are written into the captured tensors, gives that round's direct results bit
    for bit."""
    s = synth.shape(case["config"], **{k: v for k, v in case.items() if k != "config"})
    inputs = [synth.make_inputs(s, device="cuda", seed=60 + i) for i in range(3)]
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, dtlib.Weights.of(inputs[0]))
    ref = []
    for inp in inputs:
        out = rnd.round(inp.logits, inp.h0)
        ref.append(({k: v.clone() for k, v in out.items()}, rnd.ids.clone(), rnd.vals.clone()))
    torch.cuda.synchronize()
    rnd.check()
    logits, h0 = inputs[0].logits.clone(), inputs[0].h0.clone()
    graph = rnd.capture(logits, h0)
    for (ro, ri, rv), inp in zip(ref, inputs):
        logits.copy_(inp.logits)
        h0.copy_(inp.h0)
        for v in rnd.out.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        rnd.check()
        assert torch.equal(rnd.ids, ri) and torch.equal(rnd.vals, rv)
        for k in ro:
            assert torch.equal(rnd.out[k], ro[k]), k


@pytest.mark.parametrize("config", [1, 0])
def test_host_round_matches_the_device_round(dtlib, config):
    """HostRound (inputs and outputs in one pinned buffer each, one copy each way) gives the device round's outputs
    exactly, round after round."""
    inp = synth.make_inputs(config, device="cuda")
    s = inp.shape
    w = dtlib.Weights.of(inp)
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w)
    ref = {k: v.cpu() for k, v in rnd(inp.logits, inp.h0).items()}
    hr = dtlib.HostRound(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w, inp.logits.dtype)
    for _ in range(2):
        out = hr.run(inp.logits.cpu(), inp.h0.cpu())
        torch.cuda.synchronize()
        hr.check()
        for k in ref:
            assert torch.equal(ref[k], out[k]), k


def test_captured_host_round_replays_new_inputs(dtlib):
    """HostRound.capture: the graph of one host round (pinned copy in, dt_round, copy out), replayed after each round's
    inputs are written into the pinned buffers, leaves that round's device results in host_out bit for bit."""
    s = synth.shape(1)
    inputs = [synth.make_inputs(s, device="cuda", seed=80 + i) for i in range(3)]
    w = dtlib.Weights.of(inputs[0])
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w)
    refs = [{k: v.cpu() for k, v in rnd(inp.logits, inp.h0).items()} for inp in inputs]
    hr = dtlib.HostRound(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, w, inputs[0].logits.dtype)
    hr.host_logits.copy_(inputs[0].logits)
    hr.host_h0.copy_(inputs[0].h0)
    graph = hr.capture()
    torch.cuda.synchronize()
    for ref, inp in zip(refs, inputs):
        hr.host_logits.copy_(inp.logits)
        hr.host_h0.copy_(inp.h0)
        for v in hr.host_out.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        hr.check()
        for k in ref:
            assert torch.equal(ref[k], hr.host_out[k]), k


@pytest.mark.parametrize("config", [1, 2])
def test_build_stats_describe_the_launch(dtlib, config):
    """The statistics a builder launch records: its waves and expansions, and the correction rows it gathered."""
    inp = synth.make_inputs(config, device="cuda")
    s = inp.shape
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, dtlib.Weights.of(inp))
    out = rnd(inp.logits, inp.h0)
    st = dtlib.dt_build_stats_read(rnd.workspace)
    rnd.check()
    depth = out["depth"].cpu().numpy()
    assert 1 <= st["waves"] <= s.n + 16
    assert st["expansions"] >= s.B * 1 + int((depth[:, :-1] < s.max_depth).sum())  # the roots and every needed step
    assert st["gather_bytes"] > 0 and st["gather_bytes"] % (s.M * s.H * 2) == 0   # whole rows of H bf16
    assert 0 < st["gather_ns"] < st["launch_ns"] < 10_000_000
