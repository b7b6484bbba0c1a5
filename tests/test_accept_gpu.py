"""dt_accept_paths on the GPU against the CPU oracle: bit-exact accepted lengths, paths and bonus tokens, on the
trees the builder emits for every workload and on synthetic target tokens that agree with the draft at several
rates."""
import numpy as np
import pytest
import torch

from speculative_decoding_tree_top_gb300 import synth

pytestmark = pytest.mark.gpu


def check(dtlib, orc, tokens, parents, target_next):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    got = dtlib.dt_accept_paths(d(tokens), d(parents), d(target_next))
    torch.cuda.synchronize()
    want = orc.accept_paths(tokens, parents, target_next)
    for k in ("accept_len", "path", "bonus"):
        assert np.array_equal(got[k].cpu().numpy(), want[k]), k
    return want


@pytest.mark.parametrize("config", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("p_agree", [0.0, 0.6, 0.95, 1.0])
def test_accept_on_built_trees(dtlib, orc, config, p_agree):
    inp = synth.make_inputs(config, device="cuda")
    s = inp.shape
    rnd = dtlib.Round(s.B, s.K, s.V, s.M, s.n, s.max_depth, s.T, dtlib.Weights.of(inp))
    out = rnd(inp.logits, inp.h0)
    torch.cuda.synchronize()
    tok, par = out["tokens"].cpu().numpy(), out["parents"].cpu().numpy()
    tn = synth.make_target_next(tok, par, s.V, p_agree, seed=config * 10 + int(p_agree * 10))
    want = check(dtlib, orc, tok, par, tn)
    if p_agree == 1.0:  # the target follows a child wherever one exists: the walk ends at a leaf
        for b in range(s.B):
            last = want["path"][b, want["accept_len"][b] - 1]
            assert want["accept_len"][b] >= 1 and not np.any(par[b] == last)


def test_accept_edge_cases(dtlib, orc):
    # a single node, accepted or not; a chain accepted all the way; repeated tokens among siblings (earlier pop)
    check(dtlib, orc, np.array([[7]]), np.array([[-1]]), np.array([[7, 3]]))
    check(dtlib, orc, np.array([[7]]), np.array([[-1]]), np.array([[8, 3]]))
    n = 40
    chain_t = np.arange(n)[None] + 100
    chain_p = np.arange(-1, n - 1)[None]
    tn = np.concatenate([chain_t, [[5]]], axis=1)
    want = check(dtlib, orc, chain_t, chain_p, tn)
    assert want["accept_len"][0] == n and want["bonus"][0] == 5
    check(dtlib, orc, np.array([[4, 4, 9]]), np.array([[-1, -1, 1]]), np.array([[4, 9, 1, 2]]))
    # many requests (several CTAs, a partial last one)
    rng = np.random.default_rng(3)
    B, n = 37, 33
    par = np.stack([[-1] + [int(rng.integers(-1, i)) for i in range(1, n)] for _ in range(B)])
    tok = rng.integers(0, 5, size=(B, n))
    check(dtlib, orc, tok, par, rng.integers(0, 5, size=(B, n + 1)))
