"""dt_lmhead_topm on the GPU against the CPU oracle: the top-M of the full-vocabulary projection.

The kernel's logits are fp32 sums of bf16 products taken in the tensor cores' order; the oracle's are fp64. The
bar: every reported value is the fp64 logit of its reported id within TOL; the values are in descending order; the
ids equal the oracle's wherever the oracle's values leave a gap wider than 2 TOL on both sides (and at the M-th
place against the first value left out), and otherwise are a valid choice among values tied within TOL."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from speculative_decoding_tree_top_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 2e-4   # fp32 accumulation of up to 2560 products of magnitude ~0.02 (logits ~ N(0, 1)): errors ~1e-6


def check_rows(ids, vals, full, o_ids, o_vals, M):
    """ids/vals: the GPU's [R,M]; full: fp64 logits [R,V]; o_ids/o_vals: the oracle's [R,M]."""
    R, V = full.shape
    for r in range(R):
        assert np.all(np.diff(vals[r]) <= 0), r                                    # descending
        assert np.all(np.abs(full[r, ids[r]] - vals[r]) <= TOL), r                 # each value is its id's logit
        assert len(set(ids[r].tolist())) == M, r                                   # distinct ids
        assert np.all(np.abs(vals[r] - o_vals[r]) <= TOL), r                       # the sorted values agree
        order = np.lexsort((np.arange(V), -full[r]))
        nxt = full[r, order[M]] if M < V else -np.inf
        ov = o_vals[r]
        for m in range(M):
            lo = ov[m + 1] if m + 1 < M else nxt
            hi = ov[m - 1] if m > 0 else np.inf
            if hi - ov[m] > 2 * TOL and ov[m] - lo > 2 * TOL:
                assert ids[r, m] == o_ids[r, m], (r, m)


def run(dtlib, R, D, V, M, seed=4321, prep=None):
    h, w = synth.make_lmhead_inputs(R, D, V, seed=seed)
    if prep is not None:
        h, w = prep(h, w)
    hd, wd = h.cuda(), w.cuda()
    ws = dtlib.new_workspace(dtlib.dt_lmhead_workspace_bytes(R, D, V, M))
    ids, vals = dtlib.dt_lmhead_topm(hd, wd, M, workspace=ws)
    torch.cuda.synchronize()
    status = dtlib.dt_get_error(ws)
    hb, wb = synth.bits_u16(h), synth.bits_u16(w)
    return ids.cpu().numpy(), vals.cpu().numpy(), hb, wb, status


def fp64_logits(hb, wb):
    f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return f(hb) @ f(wb).T


@pytest.mark.parametrize("R,D,V,M", [
    (16, 2560, 151936, 64),    # one request of the Qwen3-4B-shaped workload: the bench case
    (1, 64, 1000, 8),          # one K block, a partial last tile, most CTAs without a tile
    (64, 128, 30000, 128),     # the most rows the tensor-memory slice takes
    (5, 192, 4096, 1),         # rows padded to 16, the arg-max
    (3, 64, 900, 900),         # M = V: the whole vocabulary in order (the bound takes every logit)
])
def test_lmhead_topm_parity(dtlib, R, D, V, M):
    ids, vals, hb, wb, status = run(dtlib, R, D, V, M)
    assert status == dtlib.Status.OK
    o_ids, o_vals = orc.lmhead_topm(hb, wb, M)
    check_rows(ids, vals, fp64_logits(hb, wb), o_ids, o_vals, M)


@pytest.mark.parametrize("R,D,V,M", [
    (65, 128, 30000, 64),      # one row past the one-launch kernel: one hidden block of 80 (rows 65..79 padding)
    (300, 192, 20000, 128),    # two hidden blocks of 256, the second partial
    (100, 64, 1000, 1000),     # M = V: the pool holds fewer than M values, the bound takes every logit
    (129, 64, 3000, 1),        # the arg-max
])
def test_lmhead_topm_blocked_parity(dtlib, R, D, V, M):
    """More rows than the tensor-memory slice takes: the blocked passes (pool, bound, filter, select)."""
    ids, vals, hb, wb, status = run(dtlib, R, D, V, M)
    assert status == dtlib.Status.OK
    o_ids, o_vals = orc.lmhead_topm(hb, wb, M)
    check_rows(ids, vals, fp64_logits(hb, wb), o_ids, o_vals, M)


def test_lmhead_topm_batched_round_shape(dtlib):
    """The batched round's projection, 64 requests x 16 block positions of the Qwen3-4B-shaped drafter (R = 1024, D =
    2560, V = 151936, M = 64). A row's top M depends on that row alone, so the oracle checks sampled rows, one in
    every hidden block and at both ends of each."""
    R, D, V, M = 1024, 2560, 151936, 64
    ids, vals, hb, wb, status = run(dtlib, R, D, V, M, seed=77)
    assert status == dtlib.Status.OK
    rows = np.array([0, 1, 255, 256, 511, 640, 767, 1023])
    o_ids, o_vals = orc.lmhead_topm(np.ascontiguousarray(hb[rows]), wb, M)
    check_rows(ids[rows], vals[rows], fp64_logits(hb[rows], wb), o_ids, o_vals, M)


def test_lmhead_topm_equal_logits_go_to_the_lower_id(dtlib):
    """Duplicated head rows in different tiles (different CTAs) give bit-equal logits: the lower id comes first."""
    def prep(h, w):
        w = w.clone()
        w[900] = w[5] = w[5] * 8            # large logits, so the pair is in every row's top M
        w[4100] = w[77] = w[77] * 8
        return h, w
    R, D, V, M = 4, 128, 5000, 16
    ids, vals, hb, wb, status = run(dtlib, R, D, V, M, prep=prep)
    assert status == dtlib.Status.OK
    for r in range(R):
        pos = {int(i): m for m, i in enumerate(ids[r])}
        for a, b in ((5, 900), (77, 4100)):
            if a in pos and b in pos:
                assert pos[a] < pos[b] and vals[r, pos[a]] == vals[r, pos[b]], (r, a, b)


def test_lmhead_topm_reports_nan(dtlib):
    """inf x 0 in the projection gives NaN logits: the status word says so and the call still returns."""
    def prep(h, w):
        h, w = h.clone(), w.clone()
        h[0, 0] = float("inf")
        w[:, 0] = 0.0
        return h, w
    *_, status = run(dtlib, 2, 64, 1000, 8, prep=prep)
    assert status == dtlib.Status.NUMERIC
    *_, status = run(dtlib, 200, 64, 1000, 8, prep=prep)   # the blocked passes
    assert status == dtlib.Status.NUMERIC


def test_lmhead_topm_blocked_equal_logits_go_to_the_lower_id(dtlib):
    """The tie rule through the blocked passes: duplicated head rows in different CTAs, 300 rows."""
    def prep(h, w):
        w = w.clone()
        w[900] = w[5] = w[5] * 8
        w[4100] = w[77] = w[77] * 8
        return h, w
    R, D, V, M = 300, 128, 5000, 16
    ids, vals, hb, wb, status = run(dtlib, R, D, V, M, prep=prep)
    assert status == dtlib.Status.OK
    o_ids, o_vals = orc.lmhead_topm(hb, wb, M)
    check_rows(ids, vals, fp64_logits(hb, wb), o_ids, o_vals, M)
    for r in range(R):
        pos = {int(i): m for m, i in enumerate(ids[r])}
        for a, b in ((5, 900), (77, 4100)):
            if a in pos and b in pos:
                assert pos[a] < pos[b] and vals[r, pos[a]] == vals[r, pos[b]], (r, a, b)
