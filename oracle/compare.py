"""GPU-vs-oracle comparison of draft trees (test infrastructure).

Rule (fp32 on the GPU, fp64 in the oracle): walk the oracle's pop order; let i* be the first pop whose gap (its
score minus the best score left in the oracle's frontier) is at most ``tol``. Before i* the two builders face the
same clear-cut decisions, so tokens, parents, depths and mask rows must be bit-identical and the scores within
``tol``. Every GPU score must be within ``tol`` of the oracle's fp64 rescoring of the GPU's own path, and from i* on
the GPU tree must satisfy the tree invariants and its sorted scores must match the oracle's within ``tol``.

Past i* the node sets are still compared, in a form ties cannot upset (``check_top_nodes``). Scores never rise along
a path (a log-softmax is at most 0, in fp32 as in fp64), so best-first pops the n highest-scoring nodes of the tree:
every node whose exact score is above the oracle's n-th score s_n is one of the oracle's pops, and every node whose
exact score is above s_n + 2 tol is one of the GPU's too (were one missing, the GPU's n pops, each scoring at least
that node's fp32 score and hence more than s_n exactly, would be n + 1 nodes above s_n with it).
"""
from __future__ import annotations

import numpy as np


def check_tree_invariants(tokens, parents, depth, scores, mask, n, max_depth):
    assert tokens.shape == (n,)
    paths = []
    for i in range(n):
        p = int(parents[i])
        assert -1 <= p < i, f"node {i}: parent {p} is not an earlier node"
        assert depth[i] == (1 if p < 0 else depth[p] + 1), f"node {i}: depth {depth[i]}"
        assert 1 <= depth[i] <= max_depth
        if p >= 0:
            assert scores[i] <= scores[p], f"node {i} scores above its parent"
        want = np.zeros(n, np.uint8)
        j = i
        while j >= 0:
            want[j] = 1
            j = int(parents[j])
        assert np.array_equal(mask[i], want), f"mask row {i} is not the ancestor closure"
        paths.append((paths[p] if p >= 0 else ()) + (int(tokens[i]),))
    assert len(set(paths)) == n, "a node appears twice"
    assert np.all(np.diff(scores) <= 0), "pops are not in best-first order"


def _paths(tokens, parents):
    paths = []
    for i, t in enumerate(tokens):
        p = int(parents[i])
        paths.append((paths[p] if p >= 0 else ()) + (int(t),))
    return paths


def check_top_nodes(gpu_tokens, gpu_parents, rescored, ora_tokens, ora_parents, ora_scores, tol):
    """The tie-robust node-set check (module docstring): nodes are token paths from the root. Every oracle node
    scoring above s_n + 2 tol is in the GPU tree, and every GPU node whose fp64 rescoring is above s_n is in the
    oracle tree. Returns the share of the oracle's nodes the first part covers."""
    gp = _paths(gpu_tokens, gpu_parents)
    op = _paths(ora_tokens, ora_parents)
    s_n = float(np.min(ora_scores))
    gset, oset = set(gp), set(op)
    covered = 0
    for path, s in zip(op, ora_scores):
        if s > s_n + 2 * tol:
            covered += 1
            assert path in gset, f"the oracle's node {path} (score {s}, n-th {s_n}) is missing from the GPU tree"
    for path, s in zip(gp, rescored):
        assert s <= s_n + 1e-9 or path in oset, f"the GPU's node {path} scores {s} above the n-th {s_n} yet is not in the oracle tree"
    return covered / len(op)


def compare_request(gpu: dict, ora: dict, rescored: np.ndarray, n: int, max_depth: int, tol: float = 1e-3,
                    struct_tol=None) -> dict:
    """gpu/ora: per-request arrays; rescored: oracle fp64 scores of the GPU's tree. Returns a small report.
    ``struct_tol`` (default ``tol``) is the gap below which two pops count as a near-tie for the structure check."""
    gaps = ora["gaps"]
    st = tol if struct_tol is None else struct_tol
    i_star = next((i for i in range(n) if gaps[i] <= st), n)
    for key in ("tokens", "parents", "depth"):
        a, b = np.asarray(gpu[key][:i_star]), np.asarray(ora[key][:i_star])
        assert np.array_equal(a, b), f"{key} differ before the first near-tie (i*={i_star}): {a} vs {b}"
    assert np.array_equal(gpu["mask"][:i_star], ora["mask"][:i_star]), "mask rows differ before the first near-tie"
    err_own = float(np.max(np.abs(gpu["scores"].astype(np.float64) - rescored)))
    assert err_own <= tol, f"GPU scores differ from the oracle's rescoring of the same tree by {err_own}"
    if i_star > 0:
        err_pre = float(np.max(np.abs(gpu["scores"][:i_star].astype(np.float64) - ora["scores"][:i_star])))
        assert err_pre <= tol, f"scores differ by {err_pre} before the first near-tie"
    check_tree_invariants(gpu["tokens"], gpu["parents"], gpu["depth"], gpu["scores"], gpu["mask"], n, max_depth)
    err_sorted = float(np.max(np.abs(np.sort(gpu["scores"].astype(np.float64)) - np.sort(ora["scores"]))))
    assert err_sorted <= tol, f"sorted scores differ by {err_sorted}"
    top = check_top_nodes(gpu["tokens"], gpu["parents"], rescored, ora["tokens"], ora["parents"], ora["scores"], tol)
    return dict(i_star=i_star, err_own=err_own, err_sorted=err_sorted, top_nodes=top)


def compare_round(gpu: dict, ora: dict, rescored: np.ndarray, n: int, max_depth: int, tol: float = 1e-3,
                  struct_tol=None) -> dict:
    """All requests of a round. gpu/ora: dicts of [B, ...] host arrays."""
    B = ora["tokens"].shape[0]
    reports = []
    for b in range(B):
        g = {k: np.asarray(gpu[k][b]) for k in ("tokens", "parents", "depth", "scores", "mask")}
        o = {k: np.asarray(ora[k][b]) for k in ("tokens", "parents", "depth", "scores", "mask", "gaps")}
        try:
            reports.append(compare_request(g, o, rescored[b], n, max_depth, tol, struct_tol))
        except AssertionError as e:
            raise AssertionError(f"request {b}: {e}") from None
    full = sum(r["i_star"] == n for r in reports)
    compared = sum(r["i_star"] for r in reports)
    return dict(requests=B, exact_structure=full, compared_pops=compared / (B * n),
                top_nodes=sum(r["top_nodes"] for r in reports) / B,
                min_i_star=min(r["i_star"] for r in reports),
                max_err_own=max(r["err_own"] for r in reports), max_err_sorted=max(r["err_sorted"] for r in reports))
