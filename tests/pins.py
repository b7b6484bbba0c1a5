"""Pins of the CPU oracle against things other than itself.

Each pin takes an oracle ctypes handle ``L`` (so the mutation test can run the same pins on deliberately broken
copies of the oracle) and raises AssertionError (or the oracle's own error) when the oracle is wrong.

What each pin leans on, outside the oracle:
  * top-M             - a full lexicographic sort of every row (numpy lexsort), i.e. brute force;
  * projection top-M  - numpy's fp64 matmul on exactly representable inputs, then the same full sort; a one-hot
                        head (closed form);
  * tree attention    - torch's scaled_dot_product_attention in fp64 with the same mask; two closed forms;
  * GRU step          - torch.nn.GRUCell in fp64 (library routine);
  * restricted softmax- with M = V it must equal torch.log_softmax over the full-vocabulary corrected row
                        computed with a dense matmul (no gather);
  * W_c = 0           - the factorised DDTree closed form: the sum of per-position log-softmaxes of the marginals;
  * best-first search - brute-force enumeration of every node of the depth-limited M-ary tree, ranked by score;
  * special cases     - M = 1 (a chain with all scores 0), max_depth = 1, n = 1;
  * golden fixtures   - hand-derived trees with closed-form scores (tests/golden);
  * invariants        - prefix closure, depths, monotone scores, ancestor-mask closure.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

from speculative_decoding_tree_top_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def widen(a):
    """Exact fp64 value of a stored array (uint16 = bf16 bit patterns, or float32)."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def tiny_inputs(seed, dtype="f32", biases=True, **kw):
    base = dict(B=1, V=512, K=4, M=6, H=16, E=24, n=12, max_depth=4, T=0.0, dtype=dtype, logit_scale=3.0,
                boost_count=8, boost_lo=2.0, boost_hi=6.0, name="pin")
    base.update(kw)
    return synth.make_inputs(synth.Shape(**base), device="cpu", seed=seed, biases=biases)


def host(inp):
    from oracle import oracle as orc
    return (synth.host_array(inp.logits), synth.host_array(inp.h0).astype(np.float64), orc.weights_of(inp))


# ----------------------------------------------------------------------------------------------------------------
def pin_topm_bruteforce(L):
    from oracle import oracle as orc
    rng = np.random.default_rng(7)
    for dtype in ("f32", "bf16"):
        B, K, V = 2, 3, 777
        x = (rng.standard_normal((B, K, V)) * 3).astype(np.float32)
        x[0, 0, :50] = 1.5                       # a block of ties
        x[0, 1, 10], x[0, 1, 11] = -0.0, 0.0     # signed zeros tie
        x[0, 1, 12:20] = 0.0
        x[1, 2, 5], x[1, 2, 6] = np.inf, -np.inf
        x[1, 0, :] = 0.25                        # a whole row of ties
        arr = x if dtype == "f32" else synth.bits_u16(torch.from_numpy(x).to(torch.bfloat16))
        full = widen(arr)
        for M in (1, 37, V):
            ids, vals = orc.topm(arr, M, L=L)
            for b in range(B):
                for k in range(K):
                    order = np.lexsort((np.arange(V), -full[b, k]))[:M]
                    assert np.array_equal(ids[b, k], order), (dtype, M, b, k)
                    assert np.array_equal(vals[b, k], full[b, k][order]), (dtype, M, b, k)


def _grucell(w_ih, w_hh, b_ih, b_hh):
    H, E = w_hh.shape[1], w_ih.shape[1]
    cell = torch.nn.GRUCell(E, H, bias=True, dtype=torch.float64)
    with torch.no_grad():
        cell.weight_ih.copy_(torch.from_numpy(widen(w_ih)))
        cell.weight_hh.copy_(torch.from_numpy(widen(w_hh)))
        cell.bias_ih.copy_(torch.from_numpy(widen(b_ih)) if b_ih is not None else torch.zeros(3 * H))
        cell.bias_hh.copy_(torch.from_numpy(widen(b_hh)) if b_hh is not None else torch.zeros(3 * H))
    return cell


def pin_gru_vs_grucell(L):
    from oracle import oracle as orc
    for dtype in ("f32", "bf16"):
        for biases in (True, False):
            inp = tiny_inputs(11, dtype=dtype, biases=biases, H=20, E=36)
            _, _, w = host(inp)
            cell = _grucell(w["w_ih"], w["w_hh"], w["b_ih"], w["b_hh"])
            rng = np.random.default_rng(3)
            for tok in (0, 17, 511):
                x = widen(w["emb"])[tok]
                h = rng.standard_normal(20)
                got = orc.gru_step(w["w_ih"], w["w_hh"], w["b_ih"], w["b_hh"], x, h, L=L)
                with torch.no_grad():
                    ref = cell(torch.from_numpy(x)[None], torch.from_numpy(h)[None])[0].numpy()
                assert np.max(np.abs(got - ref)) < 1e-12, (dtype, biases, tok, np.max(np.abs(got - ref)))


def pin_full_vocab_softmax(L):
    """M = V: the restricted log-softmax over the gathered slice equals the full conditional over the vocabulary."""
    from oracle import oracle as orc
    inp = synth.make_inputs(0, device="cpu")
    logits, _, w = host(inp)
    V = logits.shape[2]
    ids, vals = orc.topm(logits, V, L=L)
    Wc = torch.from_numpy(widen(w["w_c"]))
    rng = np.random.default_rng(5)
    for p in range(logits.shape[1]):
        h = rng.standard_normal(Wc.shape[1])
        full_row = torch.from_numpy(widen(logits)[0, p])
        for T in (0.0, 0.5, 1.0, 2.5):
            Te = T if T > 0 else 1.0
            ref = torch.log_softmax((full_row + Wc @ torch.from_numpy(h)) / Te, dim=0).numpy()
            got = orc.child_logp(w["w_c"], ids[0, p], vals[0, p], T, h, L=L)
            assert np.max(np.abs(got - ref[ids[0, p]])) < 1e-12, (p, T)
            assert abs(math.fsum(np.exp(got)) - 1.0) < 1e-12


def brute_force_nodes(ids, vals, h0, w, max_depth, T):
    """Every node of the depth-limited M-ary tree with its score, walking each path (torch, fp64)."""
    Te = T if T > 0 else 1.0
    M = ids.shape[1]
    cell = _grucell(w["w_ih"], w["w_hh"], w["b_ih"], w["b_hh"])
    Wc = torch.from_numpy(widen(w["w_c"]))
    emb = torch.from_numpy(widen(w["emb"]))
    paths = [()]
    scores = torch.zeros(1, dtype=torch.float64)
    hid = torch.from_numpy(np.asarray(h0, np.float64))[None]
    nodes = {}
    with torch.no_grad():
        for d in range(max_depth):
            cand = torch.from_numpy(ids[d].astype(np.int64))
            base = torch.from_numpy(np.asarray(vals[d], np.float64))
            logp = torch.log_softmax((base[None, :] + hid @ Wc[cand].T) / Te, dim=1)
            child_scores = (scores[:, None] + logp).reshape(-1)
            child_paths = [p + (int(t),) for p in paths for t in ids[d]]
            nodes.update(zip(child_paths, child_scores.tolist()))
            if d + 1 < max_depth:
                hid = cell(emb[cand].repeat(len(paths), 1), hid.repeat_interleave(M, dim=0))
            paths, scores = child_paths, child_scores
    return nodes


def tree_paths(tokens, parents):
    paths = []
    for i, t in enumerate(tokens):
        p = parents[i]
        paths.append((paths[p] if p >= 0 else ()) + (int(t),))
    return paths


def check_against_bruteforce(tree, nodes, n, sep=1e-9):
    paths = tree_paths(tree["tokens"], tree["parents"])
    for i, pth in enumerate(paths):
        assert pth in nodes, ("not a node of the candidate tree", pth)
        assert abs(nodes[pth] - tree["scores"][i]) < 1e-12, (i, nodes[pth], tree["scores"][i])
    ranked = sorted(nodes.items(), key=lambda kv: (-kv[1], kv[0][-1]))
    bf_scores = np.array([s for _, s in ranked])
    assert np.max(np.abs(bf_scores[:n] - np.asarray(tree["scores"]))) < 1e-12
    if len(ranked) == n or bf_scores[n - 1] - bf_scores[n] > sep:
        assert set(paths) == {p for p, _ in ranked[:n]}
    for i in range(n):
        lo_ok = i == 0 or bf_scores[i - 1] - bf_scores[i] > sep
        hi_ok = i + 1 >= len(ranked) or bf_scores[i] - bf_scores[i + 1] > sep
        if lo_ok and hi_ok:
            assert paths[i] == ranked[i][0], (i, paths[i], ranked[i][0])


def pin_bruteforce_tree(L):
    from oracle import oracle as orc
    cases = [
        (0, {}, None),                                           # the tiny oracle-check workload itself
        (21, dict(M=3, n=30, max_depth=4, T=0.5), "f32"),
        (22, dict(M=5, n=40, max_depth=3, T=1.0, H=12, E=20), "bf16"),
        (23, dict(M=4, n=60, max_depth=4, T=2.0, logit_scale=0.3), "f32"),
        (24, dict(M=2, n=14, max_depth=4, T=0.0), "bf16"),
    ]
    for seed, kw, dtype in cases:
        inp = synth.make_inputs(0, device="cpu") if dtype is None else tiny_inputs(seed, dtype=dtype, **kw)
        s = inp.shape
        logits, h0, w = host(inp)
        ids, vals = orc.topm(logits, s.M, L=L)
        tree = orc.build_trees(ids, vals, h0, w, s.n, s.max_depth, s.T, L=L)
        nodes = brute_force_nodes(ids[0], vals[0], h0[0], w, s.max_depth, s.T)
        one = {k: tree[k][0] for k in ("tokens", "parents", "scores")}
        check_against_bruteforce(one, nodes, s.n)


def pin_factorised_closed_form(L):
    """W_c = 0: each score is the sum over its path of log-softmax(top-M marginals / T) (DDTree's scoring)."""
    from oracle import oracle as orc
    for T in (0.0, 0.5, 1.0):
        inp = tiny_inputs(31, M=5, n=25, max_depth=4, T=T)
        logits, h0, w = host(inp)
        w = dict(w)
        w["w_c"] = np.zeros_like(w["w_c"])
        ids, vals = orc.topm(logits, 5, L=L)
        tree = orc.build_trees(ids, vals, h0, w, 25, 4, T, L=L)
        Te = T if T > 0 else 1.0
        marg = torch.log_softmax(torch.from_numpy(vals[0]) / Te, dim=1).numpy()   # [K, M]
        paths = tree_paths(tree["tokens"][0], tree["parents"][0])
        for i, pth in enumerate(paths):
            ref = math.fsum(marg[d][list(ids[0, d]).index(t)] for d, t in enumerate(pth))
            assert abs(ref - tree["scores"][0, i]) < 1e-12, (T, i)
        # and the factorised tree is the n best paths of the product of marginals
        nodes = {}
        for pth in _all_paths(ids[0], 4):
            nodes[pth] = math.fsum(marg[d][list(ids[0, d]).index(t)] for d, t in enumerate(pth))
        check_against_bruteforce({k: tree[k][0] for k in ("tokens", "parents", "scores")}, nodes, 25)


def pin_marginal_builder(L):
    """DDTree's marginal-scored trees: the n best nodes of the depth-limited tree under the product of the
    per-position marginals (log-softmax by torch, exhaustive enumeration), and the conditional builder at W_c = 0."""
    from oracle import oracle as orc
    cases = [(51, dict(M=5, n=25, max_depth=4, T=0.0)), (52, dict(M=3, n=30, max_depth=4, T=0.5)),
             (53, dict(M=4, n=12, max_depth=3, T=2.0, logit_scale=0.2)), (54, dict(M=1, n=4, max_depth=4, K=4))]
    for seed, kw in cases:
        inp = tiny_inputs(seed, **kw)
        s = inp.shape
        logits, h0, w = host(inp)
        ids, vals = orc.topm(logits, s.M, L=L)
        tree = orc.build_trees_marginal(ids, vals, s.n, s.max_depth, s.T, L=L)
        Te = s.T if s.T > 0 else 1.0
        marg = torch.log_softmax(torch.from_numpy(vals[0]) / Te, dim=1).numpy()
        nodes = {pth: math.fsum(marg[d][list(ids[0, d]).index(t)] for d, t in enumerate(pth))
                 for pth in _all_paths(ids[0], s.max_depth)}
        one = {k: tree[k][0] for k in ("tokens", "parents", "scores")}
        check_against_bruteforce(one, nodes, s.n)
        check_invariants(tree["tokens"][0], tree["parents"][0], tree["depth"][0], tree["scores"][0], tree["mask"][0],
                         s.n, s.max_depth)
        w0 = dict(w)
        w0["w_c"] = np.zeros_like(w["w_c"])
        cond = orc.build_trees(ids, vals, h0, w0, s.n, s.max_depth, s.T, L=L)
        for k in ("tokens", "parents", "depth", "mask"):
            assert np.array_equal(cond[k], tree[k]), k
        assert np.max(np.abs(cond["scores"] - tree["scores"])) < 1e-12


def pin_accept_paths(L):
    """The acceptance walk equals the longest root-to-node path, among all paths of the tree enumerated, whose tokens
    agree with the target's next tokens along it (greedy verification); plus the all-rejected and whole-chain cases."""
    from oracle import oracle as orc
    for trial in range(40):
        inp = tiny_inputs(70 + trial % 4, M=3, n=20, max_depth=4, T=0.5)
        logits, h0, w = host(inp)
        ids, vals = orc.topm(logits, 3, L=L)
        tree = orc.build_trees(ids, vals, h0, w, 20, 4, 0.5, L=L)
        tok, par = tree["tokens"], tree["parents"]
        tn = synth.make_target_next(tok, par, 600, p_agree=[0.0, 0.5, 0.9, 1.0][trial % 4], seed=trial)
        got = orc.accept_paths(tok, par, tn, L=L)
        best = ()
        for i in range(tok.shape[1]):   # node i's path as node indices
            nodes_on = []
            j = i
            while j >= 0:
                nodes_on.append(j)
                j = int(par[0, j])
            nodes_on.reverse()
            ok = all(int(tok[0, v]) == int(tn[0, 0 if k == 0 else 1 + nodes_on[k - 1]]) for k, v in enumerate(nodes_on))
            if ok and len(nodes_on) > len(best):
                best = tuple(nodes_on)
        assert got["accept_len"][0] == len(best), (trial, got["accept_len"][0], best)
        assert tuple(got["path"][0, :len(best)]) == best
        assert np.all(got["path"][0, len(best):] == -1)
        last = best[-1] if best else -1
        assert got["bonus"][0] == tn[0, 1 + last if best else 0]
    # nothing agrees: nothing accepted, the bonus is the target's token after the prefix
    tok = np.array([[5, 6, 7]], np.int32)
    par = np.array([[-1, 0, 1]], np.int32)
    got = orc.accept_paths(tok, par, np.array([[9, 6, 7, 8]], np.int32), L=L)
    assert got["accept_len"][0] == 0 and got["bonus"][0] == 9 and np.all(got["path"] == -1)
    # a chain the target agrees with all the way: everything accepted, the bonus comes from the leaf
    got = orc.accept_paths(tok, par, np.array([[5, 6, 7, 4]], np.int32), L=L)
    assert got["accept_len"][0] == 3 and list(got["path"][0]) == [0, 1, 2] and got["bonus"][0] == 4


def _all_paths(ids, max_depth):
    out, level = [], [()]
    for d in range(max_depth):
        level = [p + (int(t),) for p in level for t in ids[d]]
        out += level
    return out


def pin_special_cases(L):
    from oracle import oracle as orc
    # M = 1: every restricted log-softmax is exactly 0; the tree is the chain of top-1 tokens.
    inp = tiny_inputs(41, M=1, n=4, max_depth=4, K=4)
    logits, h0, w = host(inp)
    ids, vals = orc.topm(logits, 1, L=L)
    tree = orc.build_trees(ids, vals, h0, w, 4, 4, 0.0, L=L)
    assert np.array_equal(tree["tokens"][0], ids[0, :, 0])
    assert np.array_equal(tree["parents"][0], [-1, 0, 1, 2])
    assert np.array_equal(tree["depth"][0], [1, 2, 3, 4])
    assert np.all(tree["scores"][0] == 0.0)
    # max_depth = 1: the n best children of the root, by conditional log-prob then token id.
    inp = tiny_inputs(42, M=7, n=5, max_depth=1, T=0.7)
    logits, h0, w = host(inp)
    ids, vals = orc.topm(logits, 7, L=L)
    tree = orc.build_trees(ids, vals, h0, w, 5, 1, 0.7, L=L)
    z = (torch.from_numpy(vals[0, 0]) + torch.from_numpy(widen(w["w_c"])[ids[0, 0]]) @ torch.from_numpy(h0[0])) / 0.7
    lp = torch.log_softmax(z, dim=0).numpy()
    order = sorted(range(7), key=lambda m: (-lp[m], ids[0, 0, m]))[:5]
    assert np.array_equal(tree["tokens"][0], ids[0, 0, order])
    assert np.all(tree["parents"][0] == -1) and np.all(tree["depth"][0] == 1)
    assert np.max(np.abs(tree["scores"][0] - lp[order])) < 1e-12
    # n = 1: the arg-max child of the root.
    tree1 = orc.build_trees(ids, vals, h0, w, 1, 1, 0.7, L=L)
    assert tree1["tokens"][0, 0] == ids[0, 0, order[0]] and tree1["mask"][0, 0, 0] == 1


def _eval_expr(e):
    ns = {"log": math.log, "tanh": math.tanh, "sigmoid": lambda v: 1.0 / (1.0 + math.exp(-v)), "__builtins__": {}}
    return float(eval(str(e), ns))  # fixture strings are closed forms over numbers and log/tanh/sigmoid only


def _fill(spec, shape_):
    a = np.zeros(shape_, np.float32)
    if isinstance(spec, list):
        for r, c, v in spec:
            a[r, c] = _eval_expr(v)
    return a


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    V, K, H, E = g["V"], g["K"], g["H"], g["E"]
    logits = np.full((1, K, V), g["logit_default"], np.float32)
    for k, v, val in g["logits"]:
        logits[0, k, v] = _eval_expr(val)
    w = {"emb": _fill(g["emb"], (V, E)), "w_ih": _fill(g["w_ih"], (3 * H, E)), "w_hh": _fill(g["w_hh"], (3 * H, H)),
         "b_ih": _fill(g["b_ih"], (1, 3 * H))[0], "b_hh": _fill(g["b_hh"], (1, 3 * H))[0],
         "w_c": _fill(g["w_c"], (V, H))}
    h0 = np.asarray(g["h0"], np.float64)[None]
    return g, logits, h0, w


def pin_golden(L):
    from oracle import oracle as orc
    for name in ("handworked_factorised.json", "handworked_gru_path.json"):
        g, logits, h0, w = load_golden(name)
        ids, vals = orc.topm(logits, g["M"], L=L)
        tree = orc.build_trees(ids, vals, h0, w, g["n"], g["max_depth"], g["T"], L=L)
        ex = g["expected"]
        assert list(tree["tokens"][0]) == ex["tokens"], (name, tree["tokens"][0])
        assert list(tree["parents"][0]) == ex["parents"], (name, tree["parents"][0])
        assert list(tree["depth"][0]) == ex["depth"], name
        want = np.array([_eval_expr(e) for e in ex["scores"]])
        assert np.max(np.abs(tree["scores"][0] - want)) < g["tolerance"], (name, tree["scores"][0], want)


def check_invariants(tokens, parents, depth, scores, mask, n, max_depth):
    """Properties every draft tree has, whatever its arithmetic."""
    assert len(tokens) == n
    for i in range(n):
        p = parents[i]
        assert -1 <= p < i, ("not prefix-closed", i, p)
        assert depth[i] == (1 if p < 0 else depth[p] + 1), ("depth", i)
        assert 1 <= depth[i] <= max_depth
        if p >= 0:
            assert scores[i] <= scores[p], ("child scores above parent", i)
        anc = set()
        j = i
        while j >= 0:
            anc.add(j)
            j = parents[j]
        row = mask[i]
        assert all((row[j] == 1) == (j in anc) for j in range(n)), ("mask is not the ancestor closure", i)
    paths = tree_paths(tokens, parents)
    assert len(set(paths)) == n, "a node appears twice"


def pin_invariants(L):
    from oracle import oracle as orc
    for seed, kw in ((51, dict(M=8, n=60, max_depth=4)), (52, dict(M=3, n=20, max_depth=4, T=1.0)),
                     (53, dict(M=6, n=12, max_depth=2, T=0.5))):
        inp = tiny_inputs(seed, B=3, **kw)
        s = inp.shape
        logits, h0, w = host(inp)
        ids, vals = orc.topm(logits, s.M, L=L)
        tree = orc.build_trees(ids, vals, h0, w, s.n, s.max_depth, s.T, L=L)
        for b in range(s.B):
            check_invariants(tree["tokens"][b], tree["parents"][b], tree["depth"][b], tree["scores"][b],
                             tree["mask"][b], s.n, s.max_depth)
            assert np.all(np.diff(tree["scores"][b]) <= 0), "pops are not best-first"
            assert np.all(tree["gaps"][b] >= 0)


def pin_rescore(L):
    from oracle import oracle as orc
    inp = tiny_inputs(61, B=2, M=5, n=30, max_depth=4, T=0.5)
    s = inp.shape
    logits, h0, w = host(inp)
    ids, vals = orc.topm(logits, s.M, L=L)
    tree = orc.build_trees(ids, vals, h0, w, s.n, s.max_depth, s.T, L=L)
    again = orc.rescore(ids, vals, h0, w, tree["tokens"], tree["parents"], tree["depth"], s.max_depth, s.T, L=L)
    assert np.max(np.abs(again - tree["scores"])) < 1e-12
    # a tree in another valid order (breadth-first by depth) gets the brute-force path scores
    nodes = brute_force_nodes(ids[0], vals[0], h0[0], w, s.max_depth, s.T)
    chosen = sorted(nodes, key=lambda p: (len(p), p))[:s.n]
    index = {p: i for i, p in enumerate(chosen)}
    tok = np.array([[p[-1] for p in chosen]], np.int32)
    par = np.array([[index[p[:-1]] if len(p) > 1 else -1 for p in chosen]], np.int32)
    dep = np.array([[len(p) for p in chosen]], np.int32)
    sc = orc.rescore(ids[:1], vals[:1], h0[:1], w, tok, par, dep, s.max_depth, s.T, L=L)
    assert np.max(np.abs(sc[0] - [nodes[p] for p in chosen])) < 1e-12


def pin_lmhead_topm(L):
    """The top-M of the full-vocabulary projection against numpy's fp64 matmul of the widened inputs and a full
    lexicographic sort. Small-integer inputs make every dot product exact in any summation order, so the ties that
    the integers produce (and the duplicated head rows) must go to the lower id exactly. Then a one-hot head whose
    logits are the hidden values themselves, scaled per block of D vocabulary rows (a closed form)."""
    from oracle import oracle as orc
    rng = np.random.default_rng(11)
    R, D, V = 5, 96, 301
    for dtype in ("f32", "bf16"):
        h = rng.integers(-8, 9, size=(R, D)).astype(np.float32)
        w = rng.integers(-8, 9, size=(V, D)).astype(np.float32)
        w[101] = w[100]                                  # duplicated head rows: equal logits in every row
        w[250] = w[7]
        cast = (lambda a: a) if dtype == "f32" else (lambda a: synth.bits_u16(torch.from_numpy(a).to(torch.bfloat16)))
        hh, ww = cast(h), cast(w)
        full = widen(hh) @ widen(ww).T
        for M in (1, 40, V):
            ids, vals = orc.lmhead_topm(hh, ww, M, L=L)
            for r in range(R):
                order = np.lexsort((np.arange(V), -full[r]))[:M]
                assert np.array_equal(ids[r], order), (dtype, M, r)
                assert np.array_equal(vals[r], full[r][order]), (dtype, M, r)
    # one-hot head: row v of the head is 2^(v // D) e_(v mod D), so logit[r][v] = 2^(v // D) h[r][v mod D]
    D, V = 8, 40
    h = rng.standard_normal((3, D)).astype(np.float32)
    w = np.zeros((V, D), np.float32)
    for v in range(V):
        w[v, v % D] = 2.0 ** (v // D)
    ids, vals = orc.lmhead_topm(h, w, V, L=L)
    expect = np.array([[2.0 ** (v // D) * float(h[r, v % D]) for v in range(V)] for r in range(3)])
    for r in range(3):
        order = np.lexsort((np.arange(V), -expect[r]))
        assert np.array_equal(ids[r], order) and np.array_equal(vals[r], expect[r][order]), r


def _random_tree_mask(rng, B, n):
    """Ancestor masks of random prefix-closed trees (each node's parent precedes it; -1 = a child of the root)."""
    mask = np.zeros((B, n, n), np.uint8)
    for b in range(B):
        par = [-1] + [int(rng.integers(-1, i)) for i in range(1, n)]
        for i in range(n):
            j = i
            while j >= 0:
                mask[b, i, j] = 1
                j = par[j]
    return mask


def pin_tree_attention(L):
    """The verify pass's tree attention against torch's scaled_dot_product_attention in fp64 (the same boolean mask:
    every prefix key, and the tree keys of the node's ancestors and itself; the key/value heads repeated for the
    grouped query heads); then two closed forms: with no prefix and a diagonal mask every node sees only itself (out
    = its own value row), and with q = 0 all visible keys weigh the same (out = the mean of their value rows)."""
    from oracle import oracle as orc
    rng = np.random.default_rng(5)
    B, n, Lp, Hq, Hkv, d = 2, 7, 19, 4, 2, 16
    G, T = Hq // Hkv, Lp + n
    for dtype in ("f32", "bf16"):
        q = rng.standard_normal((B, n, Hq, d)).astype(np.float32)
        k = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
        v = rng.standard_normal((B, Hkv, T, d)).astype(np.float32)
        mask = _random_tree_mask(rng, B, n)
        cast = (lambda a: a) if dtype == "f32" else (lambda a: synth.bits_u16(torch.from_numpy(a).to(torch.bfloat16)))
        qq, kk, vv = cast(q), cast(k), cast(v)
        scale = 0.37
        out = orc.tree_attention(qq, kk, vv, mask, scale, L=L)
        qt = torch.from_numpy(widen(qq)).permute(0, 2, 1, 3)                       # [B,Hq,n,d]
        kt = torch.from_numpy(widen(kk)).repeat_interleave(G, dim=1)               # [B,Hq,T,d]
        vt = torch.from_numpy(widen(vv)).repeat_interleave(G, dim=1)
        am = torch.ones((B, 1, n, T), dtype=torch.bool)
        am[:, 0, :, Lp:] = torch.from_numpy(mask.astype(bool))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, scale=scale)
        assert np.max(np.abs(out - ref.permute(0, 2, 1, 3).numpy())) < 1e-12, dtype
    # no prefix, diagonal mask: each node's output is its own value row
    q = rng.standard_normal((1, n, Hq, d)).astype(np.float32)
    k = rng.standard_normal((1, Hkv, n, d)).astype(np.float32)
    v = rng.standard_normal((1, Hkv, n, d)).astype(np.float32)
    out = orc.tree_attention(q, k, v, np.eye(n, dtype=np.uint8)[None], 1.0, L=L)
    for h in range(Hq):
        assert np.array_equal(out[0, :, h], v[0, h // G].astype(np.float64)), h
    # q = 0: every visible key weighs the same
    mask = _random_tree_mask(rng, 1, n)
    k = rng.standard_normal((1, Hkv, Lp + n, d)).astype(np.float32)
    v = rng.standard_normal((1, Hkv, Lp + n, d)).astype(np.float32)
    out = orc.tree_attention(np.zeros((1, n, Hq, d), np.float32), k, v, mask, 0.5, L=L)
    for i in range(n):
        vis = list(range(Lp)) + [Lp + t for t in range(n) if mask[0, i, t]]
        for h in range(Hq):
            assert np.max(np.abs(out[0, i, h] - v[0, h // G, vis].astype(np.float64).mean(0))) < 1e-12, (i, h)


ALL_PINS = [pin_topm_bruteforce, pin_gru_vs_grucell, pin_full_vocab_softmax, pin_golden, pin_special_cases,
            pin_factorised_closed_form, pin_bruteforce_tree, pin_invariants, pin_rescore, pin_marginal_builder,
            pin_accept_paths, pin_lmhead_topm, pin_tree_attention]
