"""The seeded input generator: deterministic, the configured shapes and dtypes, distinct boosted ids."""
import torch

from speculative_decoding_tree_top_gb300 import synth


def test_deterministic_and_seeded():
    a = synth.make_inputs(0)
    b = synth.make_inputs(0)
    c = synth.make_inputs(0, seed=99)
    for k in ("logits", "h0", "w_ih", "w_hh", "b_ih", "b_hh", "emb", "w_c"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
        assert not torch.equal(getattr(a, k), getattr(c, k)), k
    assert torch.equal(synth.make_logits(0), a.logits)


def test_config_shapes():
    for i, cfg in synth.CONFIGS.items():
        s = synth.shape(i)
        assert (s.B, s.V, s.K, s.M, s.n) == (cfg["B"], cfg["V"], cfg["K"], cfg["M"], cfg["n"])
        assert 1 <= s.max_depth <= s.K and s.H % 8 == 0 and s.E % 8 == 0
    small = synth.make_inputs(2, V=4096, E=64, H=32, B=3)
    assert small.logits.dtype == torch.bfloat16 and small.logits.shape == (3, 16, 4096)
    assert small.w_ih.shape == (96, 64) and small.w_c.shape == (4096, 32) and small.h0.dtype == torch.float32


def test_boosted_ids_are_distinct():
    ids = synth._distinct_ids(50, 16, 40, "cpu", 5)
    assert ids.shape == (50, 16)
    for row in ids.tolist():
        assert len(set(row)) == 16 and all(0 <= v < 40 for v in row)
    s = synth.shape(0)
    x = synth.make_logits(0)
    # the 16 boosted ids of each position sit well above the N(0, 3^2) bulk
    assert (x[0] > 4.0).sum(dim=1).min() >= 10
    assert s.boost_count == 16
