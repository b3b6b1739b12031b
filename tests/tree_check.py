"""Structural comparison of a DominoTree built on the GPU with the oracle's.

The parity bar for trees: node ids, parents and depths bit-exact, scores within
SCORE_TOL. A mismatch is excused only where the oracle itself shows that a
different tree is an equally valid result of the same arithmetic done in a
slightly different rounding order:

  (a) the pop at the mismatching node is an oracle near tie: the popped key
      and the next key of the oracle's heap differ by less than NEAR_TIE; or
  (b) a candidate set C_t that the mismatching nodes depend on (the sets of
      every depth up to the deeper of the two nodes) really differs between
      the GPU and the oracle, and the oracle's top-M boundary gap at that
      depth is below NEAR_TIE.

Anything else fails. After an excused mismatch the two trees diverge, so the
comparison of that request stops there and the request is counted as a near
tie. Imports numpy only, so the checker itself is tested on the CPU.
"""
from __future__ import annotations

import numpy as np

NEAR_TIE = 1e-3
SCORE_TOL = 2e-3


def _same_set(a, b) -> bool:
    a = [int(x) for x in np.asarray(a).ravel() if x >= 0]
    b = [int(x) for x in np.asarray(b).ravel() if x >= 0]
    return sorted(a) == sorted(b)


def compare_tree(g, o, b, N, gpu_cands=None, score_tol=SCORE_TOL):
    """Compare request b of a GPU tree g = (token, parent, depth, score) arrays
    [batch, N+1] with the oracle's tree dict o (tree_build output, which
    carries pop_margin, cand_gap and cands [batch, P, M]). gpu_cands
    [batch, P, M] are the candidate ids the GPU selected from its own L_base
    (None: taken to equal the oracle's). Returns "exact" or "near_tie"; raises
    AssertionError on any mismatch the rules above do not excuse."""
    gt, gp, gd, gs = (np.asarray(x) for x in g)
    ot, op, od, os_ = (np.asarray(o[k]) for k in ("node_token", "node_parent", "node_depth", "node_score"))
    oc = np.asarray(o["cands"])
    gc = oc if gpu_cands is None else np.asarray(gpu_cands)
    P = oc.shape[1]
    for k in range(N + 1):
        same = gt[b, k] == ot[b, k] and gp[b, k] == op[b, k] and gd[b, k] == od[b, k]
        if same:
            if ot[b, k] >= 0:
                assert abs(float(gs[b, k]) - float(os_[b, k])) < score_tol, (
                    f"tree score b={b} node {k}: gpu {float(gs[b, k])!r} oracle {float(os_[b, k])!r}")
            continue
        why = f"gpu ({gt[b, k]},{gp[b, k]},{gd[b, k]}) oracle ({ot[b, k]},{op[b, k]},{od[b, k]})"
        if float(o["pop_margin"][b, k]) < NEAR_TIE:
            return "near_tie"
        deepest = int(max(gd[b, k], od[b, k]))
        for t in range(min(max(deepest, 0), P)):
            if float(o["cand_gap"][b, t]) < NEAR_TIE and not _same_set(gc[b, t], oc[b, t]):
                return "near_tie"
        raise AssertionError(f"tree mismatch b={b} node {k}: {why}, pop margin "
                             f"{float(o['pop_margin'][b, k]):.3g}, no candidate set differs at a near tie")
    return "exact"


def compare_trees(g, o, N, requests, gpu_cands=None, score_tol=SCORE_TOL):
    """compare_tree over several requests (indices into both g and o).
    Returns (exact, near_tie) counts."""
    res = [compare_tree(g, o, b, N, gpu_cands, score_tol) for b in requests]
    return res.count("exact"), res.count("near_tie")
