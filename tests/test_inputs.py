"""The seeded input generator: deterministic, the configured shapes and dtypes, distinct boosted ids, and the recipe's
distributions and bf16 rounding as stated."""
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


def test_recipe_statistics_and_bf16_rounding():
    """The recipe's distributions (standard deviations as stated), h0 kept fp32, and bf16 tensors that are exactly the
    fp32 draws rounded to nearest even."""
    kw = dict(V=8192, E=256, H=128, B=4)
    b = synth.make_inputs(2, **kw)
    f = synth.make_inputs(2, dtype="f32", **kw)
    s = b.shape
    for k in ("w_ih", "w_hh", "b_ih", "b_hh", "emb", "w_c"):
        assert getattr(b, k).dtype == torch.bfloat16 and getattr(f, k).dtype == torch.float32, k
        assert torch.equal(getattr(f, k).to(torch.bfloat16), getattr(b, k)), k   # one draw, rounded
    assert torch.equal(f.logits.to(torch.bfloat16), b.logits)
    assert b.h0.dtype == torch.float32 and torch.equal(b.h0, f.h0)
    want = {"w_ih": 1 / s.E ** 0.5, "w_hh": 1 / s.H ** 0.5, "b_ih": 1 / s.H ** 0.5, "b_hh": 1 / s.H ** 0.5,
            "emb": 0.02, "w_c": 0.1, "h0": 1.0}
    for k, sd in want.items():
        x = getattr(f, k).double()
        tol = 0.15 if x.numel() < 2000 else 0.03
        assert abs(x.std().item() / sd - 1) < tol and abs(x.mean().item()) < 4 * sd / x.numel() ** 0.5 + 1e-12, k
    # logits: the bulk is N(0, logit_scale^2); each row carries boost_count ids raised by U(boost_lo, boost_hi)
    rows = f.logits.reshape(-1, s.V).double()
    assert abs(rows.std(dim=1).median().item() / s.logit_scale - 1) < 0.05
    raised = (rows - synth._normal((s.B, s.K, s.V), s.logit_scale, "cpu", 1234 + 200, "logits").reshape(-1, s.V)
              .double())
    assert torch.all((raised != 0).sum(dim=1) == s.boost_count)
    nz = raised[raised != 0]
    assert nz.min().item() >= s.boost_lo - 1e-5 and nz.max().item() <= s.boost_hi + 1e-5
