"""Plants one plausible mistake at a time in a copy of the oracle (on the CPU) and checks that the pins catch it.

Each mutant is the oracle source with one substring replaced; it is compiled to a temporary library and run
through the pin suite. A mutant that passes every pin would mean the pins cannot tell that mistake apart.
"""
import os
import subprocess

import pytest

import pins
from oracle import compare
from oracle import oracle as orc

MUTANTS = {
    "topm-order-reversed": ("if (v[a] != v[b]) return v[a] > v[b];", "if (v[a] != v[b]) return v[a] < v[b];"),
    "topm-id-tiebreak-reversed": ("    return a < b;\n  });", "    return a > b;\n  });"),
    "gru-drops-b_hh": ("double c = bias(w.b_hh, w.dtype, row);", "double c = 0.0;"),
    "gru-reset-gate-wrong-row": ("in_side[2] + r * hid_side[2]", "in_side[2] + r * hid_side[1]"),
    "gru-update-gate-swapped": ("out[k] = (1.0 - u) * g + u * h[k];", "out[k] = u * g + (1.0 - u) * h[k];"),
    "gru-sigmoid-sign": ("1.0 / (1.0 + std::exp(-(in_side[0] + hid_side[0])))",
                         "1.0 / (1.0 + std::exp(in_side[0] + hid_side[0]))"),
    "correction-columns-reversed": ("static_cast<size_t>(ids[m]) * H + k] ", "XX"),
    "correction-after-temperature": ("z[m] = (base[m] + s) / T_eff;", "z[m] = base[m] / T_eff + s;"),
    "softmax-drops-normaliser": ("logp[m] = (z[m] - mx) - lse;", "logp[m] = z[m] - mx;"),
    "position-off-by-one": ("child_logp(w, ids + static_cast<size_t>(d) * M, vals + static_cast<size_t>(d) * M,",
                            "child_logp(w, ids + static_cast<size_t>(d > 0 ? d - 1 : 0) * M, "
                            "vals + static_cast<size_t>(d > 0 ? d - 1 : 0) * M,"),
    "heap-token-tiebreak-reversed": ("if (a.token != b.token) return a.token > b.token;",
                                     "if (a.token != b.token) return a.token < b.token;"),
    "heap-seq-tiebreak-reversed": ("return a.seq > b.seq;", "return a.seq < b.seq;"),
    "hidden-state-not-carried": ("const double* hp = u.parent < 0 ? h0 : &hs[static_cast<size_t>(u.parent) * H];",
                                 "const double* hp = h0;"),
    "score-not-cumulative": ("frontier.push(Cand{score + logp[m],", "frontier.push(Cand{logp[m],"),
    "mask-self-only": ("for (int j = i; j >= 0; j = parents[j]) mask", "for (int j = i; j == i; j = parents[j]) mask"),
    "marginal-drops-temperature": ("marg[static_cast<size_t>(d) * M + m] = (v[m] / T_eff - mx) - lse;",
                                   "marg[static_cast<size_t>(d) * M + m] = (v[m] - mx) - lse;"),
    "marginal-position-off-by-one": ("expand(i, u.depth, u.score);", "expand(i, u.depth > 1 ? u.depth - 1 : 0, u.score);"),
    "accept-target-index-off-by-one": ("want = target_next[1 + next];", "want = target_next[next];"),
    "accept-root-token-skipped": ("int cur = -1, len = 0, want = target_next[0];",
                                  "int cur = -1, len = 0, want = target_next[1];"),
    "lmhead-drops-last-term": ("for (int k = 0; k < D; ++k) acc += h[k] * load(w_head,",
                               "for (int k = 0; k + 1 < D; ++k) acc += h[k] * load(w_head,"),
    "lmhead-head-transposed": ("load(w_head, wdtype, static_cast<size_t>(v) * D + k)",
                               "load(w_head, wdtype, (static_cast<size_t>(k) * V + v) % (static_cast<size_t>(V) * D))"),
    "lmhead-hidden-row-0": ("h[k] = load(hidden, hdtype, static_cast<size_t>(r) * D + k);",
                            "h[k] = load(hidden, hdtype, static_cast<size_t>(k));"),
    "attention-mask-transposed": ("mask[(static_cast<size_t>(b) * n + i) * n + (j - L)]",
                                  "mask[(static_cast<size_t>(b) * n + (j - L)) * n + i]"),
    "attention-kv-head-interleaved": ("const int kvh = h / G;", "const int kvh = h % Hkv;"),
    "attention-drops-scale": ("sc[j] = scale * dot;", "sc[j] = dot;"),
    "embedding-of-parent": ("load(w.emb, w.dtype, static_cast<size_t>(u.token) * E + e)",
                            "load(w.emb, w.dtype, static_cast<size_t>(u.parent < 0 ? u.token : tokens[u.parent]) * E + e)"),
}


def _mutant_source(name):
    src = orc.SRC.read_text()
    old, new = MUTANTS[name]
    if name == "correction-columns-reversed":
        old = "load(w.w_c, w.dtype, static_cast<size_t>(ids[m]) * H + k)"
        new = "load(w.w_c, w.dtype, static_cast<size_t>(ids[m]) * H + (H - 1 - k))"
    assert src.count(old) >= 1, f"mutation site of {name} not found"
    return src.replace(old, new)


def _compile(name, tmp_path):
    src = tmp_path / "mutant.cpp"
    src.write_text(_mutant_source(name))
    out = tmp_path / "libmutant.so"
    cmd = orc.compile_command(src, out)
    cmd[1] = "-O1"
    subprocess.run(cmd, check=True)
    return orc.load(out)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    L = _compile(name, tmp_path)
    caught = None
    for pin in pins.ALL_PINS:
        try:
            pin(L)
        except (AssertionError, orc.OracleError, ValueError, IndexError) as e:
            caught = (pin.__name__, type(e).__name__)
            break
    assert caught is not None, f"no pin detects the planted mistake {name!r}"


# The mutants that change the trees themselves: the GPU-vs-oracle rule (oracle/compare.py) must reject their trees,
# as it would a kernel's that made the same mistake (the tie-break mutants are left to the golden trees: ties are
# rare on random inputs).
TREE_MUTANTS = ["gru-drops-b_hh", "gru-reset-gate-wrong-row", "gru-update-gate-swapped", "gru-sigmoid-sign",
                "correction-columns-reversed", "correction-after-temperature", "softmax-drops-normaliser",
                "position-off-by-one", "hidden-state-not-carried", "score-not-cumulative", "mask-self-only",
                "embedding-of-parent"]


@pytest.mark.parametrize("name", TREE_MUTANTS)
def test_parity_rule_rejects_mutant_trees(name, tmp_path):
    L = _compile(name, tmp_path)
    inp = pins.tiny_inputs(5, dtype="bf16", B=4, M=6, n=16, max_depth=4, T=0.5)
    s = inp.shape
    logits, h0, w = pins.host(inp)
    ids, vals = orc.topm(logits, s.M)
    ora = orc.build_trees(ids, vals, h0, w, s.n, s.max_depth, s.T)
    bad = orc.build_trees(ids, vals, h0, w, s.n, s.max_depth, s.T, L=L)
    resc = orc.rescore(ids, vals, h0, w, bad["tokens"], bad["parents"], bad["depth"], s.max_depth, s.T)
    compare.compare_round(ora, ora, orc.rescore(ids, vals, h0, w, ora["tokens"], ora["parents"], ora["depth"],
                                                s.max_depth, s.T), s.n, s.max_depth)  # the rule accepts the oracle
    with pytest.raises(AssertionError):
        compare.compare_round(bad, ora, resc, s.n, s.max_depth)
    # and past the first near-tie too (no bit-exact prefix at all), with the mutant's own scores or with its tree
    # given the true scores, so that only the tree's shape can tell
    relabelled = dict(bad, scores=resc)
    for tree in (bad, relabelled):
        with pytest.raises(AssertionError):
            compare.compare_round(tree, ora, resc, s.n, s.max_depth, struct_tol=float("inf"))
