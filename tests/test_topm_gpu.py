"""dt_topm on the GPU against the CPU oracle: bit-exact ids and values (integer work)."""
import numpy as np
import pytest
import torch

from speculative_decoding_tree_top_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["cluster", "lists"])
def topm_kernel(dtlib, request):
    """Every case runs twice: small launches through the one-cluster-per-row kernel, and with that kernel switched off
    (per-chunk candidate lists and the row selection). Large launches take the lists either way."""
    dtlib.dt_set_topm_cluster(request.param == "cluster")
    yield request.param
    dtlib.dt_set_topm_cluster(True)


def _host(t):
    return synth.host_array(t)


def _check(dtlib, orc, logits, M):
    ids, vals = dtlib.dt_topm(logits, M)
    torch.cuda.synchronize()
    o_ids, o_vals = orc.topm(_host(logits), M)
    g_ids, g_vals = ids.cpu().numpy(), vals.cpu().numpy()
    bad = np.argwhere(g_ids != o_ids)
    assert bad.size == 0, f"ids differ at {bad[:5].tolist()}"
    assert np.array_equal(g_vals.astype(np.float64), o_vals)
    return ids, vals


@pytest.mark.parametrize("config", [0, 1, 2, 3, 4])
def test_topm_parity_workloads(dtlib, orc, config):
    s = synth.shape(config)
    logits = synth.make_logits(config, device="cuda")
    _check(dtlib, orc, logits, s.M)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,K,V,M", [(2, 3, 1000, 17), (1, 2, 1001, 8), (2, 2, 8191, 64), (1, 3, 8193, 64),
                                     (1, 2, 16384, 128), (1, 2, 700, 700), (1, 1, 5000, 1024), (3, 2, 40000, 1),
                                     (1, 2, 8, 3), (2, 2, 100003, 256), (1, 4, 8200, 256), (2, 3, 16392, 100),
                                     (1, 1, 2048, 256), (1, 16, 151936, 64)])
def test_topm_ragged_shapes(dtlib, orc, dtype, B, K, V, M):
    g = torch.Generator(device="cuda").manual_seed(B * 7919 + V)
    x = (torch.randn((B, K, V), generator=g, device="cuda") * 3).to(dtype)
    _check(dtlib, orc, x, M)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_topm_ties_zeros_infinities(dtlib, orc, dtype):
    V = 3 * 8192 + 77
    x = torch.randn((1, 6, V), device="cuda") * 2
    x[0, 0] = 0.5                                   # a whole row of ties: the lowest ids win
    x[0, 1, ::2] = -0.0
    x[0, 1, 1::2] = 0.0                             # signed zeros tie
    x[0, 2, 100] = float("inf")
    x[0, 2, 200] = float("-inf")
    x[0, 2, 9000] = float("inf")
    x[0, 3] = torch.round(x[0, 3] * 4) / 4          # heavy ties everywhere
    x[0, 4, :] = -1.0
    x[0, 4, 8192 * 2 + 5:] = 3.0                    # all the winners sit in the last chunks
    x[0, 5] = torch.where(torch.arange(V, device="cuda") % 8192 < 40, 7.0, -7.0)  # 40 winners in every chunk
    x = x.to(dtype)
    for M in (1, 64, 200):
        ids, vals = _check(dtlib, orc, x, M)
    row0 = ids[0, 0].cpu().numpy()
    assert np.array_equal(row0, np.arange(200))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_topm_rows_in_whole_groups(dtlib, orc, dtype):
    """The same extremes with a row length that is a whole number of 16-byte groups (the cluster kernel's domain):
    slices of ties, rows of ties, winners crowded into one slice, a slice of -inf."""
    V = 3 * 8192 + 80
    x = torch.randn((1, 7, V), device="cuda") * 2
    x[0, 0] = 0.5
    x[0, 1, ::2] = -0.0
    x[0, 1, 1::2] = 0.0
    x[0, 2, 100] = float("inf")
    x[0, 2, 200] = float("-inf")
    x[0, 2, 9000] = float("inf")
    x[0, 3] = torch.round(x[0, 3] * 4) / 4
    x[0, 4, :] = -1.0
    x[0, 4, V - 300:] = 3.0                          # all the winners in the last slice
    x[0, 5] = torch.where(torch.arange(V, device="cuda") % 3082 < 40, 7.0, -7.0)  # 40 winners in every slice
    x[0, 6, : V // 2] = float("-inf")                # half the row at -inf
    x = x.to(dtype)
    for M in (1, 64, 200, 256):
        ids, _ = _check(dtlib, orc, x, M)
        assert np.array_equal(ids[0, 0].cpu().numpy(), np.arange(M))


def test_topm_merge_with_many_candidates(dtlib, orc):
    """A row whose chunk lists all reach the merge bound: the merge takes its exact (bisection) path."""
    V, M = 19 * 8192, 64
    x = torch.full((1, 1, V), -5.0, device="cuda")
    val = 100.0
    for c in range(19):
        for j in range(M - 1):
            x[0, 0, c * 8192 + 10 * j + 3] = val
            val += 1.0
    x[0, 0, 1] = 50.0   # chunk 0's M-th entry is the smallest "high" value, so every high value reaches the bound
    _check(dtlib, orc, x, M)


def test_topm_deterministic(dtlib):
    x = synth.make_logits(2, device="cuda")
    a = [t.clone() for t in dtlib.dt_topm(x, 64)]
    b = dtlib.dt_topm(x, 64)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_topm_nan_is_reported(dtlib):
    x = torch.randn((1, 2, 4096), device="cuda").to(torch.bfloat16)
    x[0, 1, 77] = float("nan")
    ws = dtlib.new_workspace(dtlib.dt_topm_workspace_bytes(1, 2, 4096, 8))
    ids, _ = dtlib.dt_topm(x, 8, workspace=ws)
    assert dtlib.dt_get_error(ws) == dtlib.Status.NUMERIC
    assert dtlib.dt_get_error(ws) == dtlib.Status.OK      # read-and-clear
    assert int(ids.min()) >= 0 and int(ids.max()) < 4096


def test_topm_empty_batch(dtlib):
    x = torch.empty((0, 4, 1024), device="cuda", dtype=torch.bfloat16)
    ids, vals = dtlib.dt_topm(x, 8)
    assert ids.shape == (0, 4, 8)


# bf16 rows whose length is a multiple of 8 logits with M <= 128 take the streaming kernel (persistent CTAs, a
# running threshold per row segment); the cases below reach its buffer-overflow, exact-bisection, compaction and
# split-row merge paths.
@pytest.mark.parametrize("M", [1, 64, 128])
def test_topm_streaming_ties_and_extremes(dtlib, orc, M):
    V = 3 * 16384 + 80
    x = torch.randn((1, 7, V), device="cuda") * 2
    x[0, 0] = 0.5                                   # all ties: the first stage overflows, the exact path decides
    x[0, 1, ::2] = -0.0
    x[0, 1, 1::2] = 0.0
    x[0, 2, 100] = float("inf")
    x[0, 2, 20000] = float("-inf")
    x[0, 3] = torch.round(x[0, 3] * 4) / 4          # heavy ties everywhere
    x[0, 4, :] = -1.0
    x[0, 4, 16384 * 2 + 5:] = 3.0                   # all the winners in the last stage
    stage = torch.arange(V, device="cuda") // 16384
    x[0, 5] = torch.randn(V, device="cuda") + 10.0 * stage   # every stage beats all earlier ones
    x[0, 6] = torch.where(torch.arange(V, device="cuda") % 16384 < 40, 7.0, -7.0)
    ids, _ = _check(dtlib, orc, x.to(torch.bfloat16), M)
    assert np.array_equal(ids[0, 0].cpu().numpy(), np.arange(M))


def test_topm_streaming_rows_split_across_ctas(dtlib, orc):
    """160 rows of 3 stages over at most 2 CTAs per SM: segments start and end inside rows."""
    g = torch.Generator(device="cuda").manual_seed(11)
    x = (torch.randn((4, 40, 40000), generator=g, device="cuda") * 3).to(torch.bfloat16)
    _check(dtlib, orc, x, 64)
