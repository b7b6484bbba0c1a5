"""The comparison helper's node-set check (oracle/compare.py, check_top_nodes) on the CPU. Best-first trees grown on
scores perturbed by less than the tolerance, as an fp32 builder's are, must pass it against the oracle's tree. Trees
with a wrong token, a wrong parent or a foreign node must fail it."""
import heapq

import numpy as np
import pytest

import pins
from oracle import compare

TOL = 1e-3
CASES = [
    (41, dict(M=4, n=30, max_depth=4, T=0.5)),
    (42, dict(M=5, n=40, max_depth=3, T=1.0, logit_scale=0.3)),  # flat logits: many near-ties
    (43, dict(M=3, n=25, max_depth=4, T=0.0, logit_scale=0.2, boost_count=0)),
    (44, dict(M=6, n=12, max_depth=2, T=2.0)),
]


def noisy_best_first(nodes, ids, n, max_depth, delta, rng):
    """Best-first over the brute-force scores with every path step's log-probability moved by at most `delta` and
    kept <= 0 (scores never rise along a path, as in the GPU's fp32). Returns the n pops' tokens, parents and exact
    scores."""
    g = {(): 0.0}
    heap, seq = [], 0

    def push_children(path):
        nonlocal seq
        d = len(path)
        if d >= max_depth:
            return
        for t in ids[d]:
            c = path + (int(t),)
            step = nodes[c] - (nodes[path] if path else 0.0)
            g[c] = g[path] + min(0.0, step + rng.uniform(-delta, delta))
            heapq.heappush(heap, (-g[c], seq, c))
            seq += 1

    push_children(())
    pops, index = [], {}
    while len(pops) < n:
        c = heapq.heappop(heap)[2]
        index[c] = len(pops)
        pops.append(c)
        if len(pops) < n:
            push_children(c)
    tokens = np.array([c[-1] for c in pops])
    parents = np.array([index[c[:-1]] if len(c) > 1 else -1 for c in pops])
    return tokens, parents, np.array([nodes[c] for c in pops])


def oracle_case(orc, seed, kw):
    inp = pins.tiny_inputs(seed, **kw)
    s = inp.shape
    logits, h0, w = pins.host(inp)
    ids, vals = orc.topm(logits, s.M)
    tree = orc.build_trees(ids, vals, h0, w, s.n, s.max_depth, s.T)
    ora = {k: np.asarray(tree[k][0]) for k in ("tokens", "parents", "scores")}
    nodes = pins.brute_force_nodes(ids[0], vals[0], h0[0], w, s.max_depth, s.T)
    return s, ids[0], ora, nodes


@pytest.mark.parametrize("seed,kw", CASES)
def test_noisy_best_first_trees_pass(orc, seed, kw):
    s, ids, ora, nodes = oracle_case(orc, seed, kw)
    rng = np.random.default_rng(seed)
    reordered = 0
    for delta in (TOL / 8, TOL / 2 / s.max_depth):  # at most TOL / 2 off at any depth
        for _ in range(10):
            tokens, parents, exact = noisy_best_first(nodes, ids, s.n, s.max_depth, delta, rng)
            compare.check_top_nodes(tokens, parents, exact, ora["tokens"], ora["parents"], ora["scores"], TOL)
            reordered += not (np.array_equal(tokens, ora["tokens"]) and np.array_equal(parents, ora["parents"]))
    # the exact best-first tree is the oracle's, and passes with full coverage of the clear nodes
    tokens, parents, exact = noisy_best_first(nodes, ids, s.n, s.max_depth, 0.0, rng)
    assert compare.check_top_nodes(tokens, parents, exact, ora["tokens"], ora["parents"], ora["scores"], TOL) > 0


@pytest.mark.parametrize("seed", range(6))
def test_tie_heavy_trees_pass(seed):
    """Synthetic trees whose path steps come from a few values 1e-4 apart (exact and near ties everywhere): the
    exact best-first tree against noisy ones, which reorder and swap nodes at every near-tie."""
    rng = np.random.default_rng(100 + seed)
    M, D, n = 4, 4, 40
    ids = np.array([rng.permutation(50)[:M] for _ in range(D)])
    steps = np.array([-0.2, -0.2001, -0.2003, -0.5, -0.5002, -1.0])
    nodes, paths = {}, [()]
    for d in range(D):
        nxt = []
        for pth in paths:
            for t in ids[d]:
                c = pth + (int(t),)
                nodes[c] = (nodes[pth] if pth else 0.0) + float(rng.choice(steps))
                nxt.append(c)
        paths = nxt
    ref_t, ref_p, ref_s = noisy_best_first(nodes, ids, n, D, 0.0, rng)
    reordered, covered = 0, []
    for _ in range(40):
        tokens, parents, exact = noisy_best_first(nodes, ids, n, D, TOL / 2 / D, rng)
        covered.append(compare.check_top_nodes(tokens, parents, exact, ref_t, ref_p, ref_s, TOL))
        reordered += not (np.array_equal(tokens, ref_t) and np.array_equal(parents, ref_p))
    assert reordered > 0 and min(covered) > 0


@pytest.mark.parametrize("seed,kw", CASES)
def test_wrong_trees_fail(orc, seed, kw):
    s, ids, ora, nodes = oracle_case(orc, seed, kw)
    tok, par, sc = ora["tokens"], ora["parents"], ora["scores"]
    paths = compare._paths(tok, par)

    def fails(t, p, resc):
        with pytest.raises(AssertionError):
            compare.check_top_nodes(t, p, resc, tok, par, sc, TOL)

    foreign = int(ids.max()) + 1  # a token that is no candidate at any position
    # the best node's token replaced: its path, and those of its descendants, leave the tree
    t2 = tok.copy()
    t2[0] = foreign
    fails(t2, par, sc)
    # a clear node of depth >= 2 hung under another node of its parent's depth
    pset = set(paths)
    k, alt = next(((i, j) for i in range(s.n) if par[i] >= 0 and sc[i] > sc.min() + 2 * TOL for j in range(i)
                   if j != par[i] and len(paths[j]) == len(paths[par[i]]) and paths[j] + (int(tok[i]),) not in pset),
                  (None, None))
    if alt is not None:
        p2 = par.copy()
        p2[k] = alt
        fails(tok, p2, sc)
    # the last pop (a leaf at the n-th score, which the first part does not cover) swapped for a node outside the
    # oracle's tree whose rescoring clears the n-th score
    t3, r3 = tok.copy(), sc.copy()
    t3[-1] = foreign
    r3[-1] = sc.min() + 0.5
    fails(t3, par, r3)
    # and with its true, lower score the same swap passes: below the n-th score either tree may hold either node
    r3[-1] = sc.min() - 0.5
    compare.check_top_nodes(t3, par, r3, tok, par, sc, TOL)
    assert k is not None and alt is not None or s.max_depth < 2 or s.n < 8
