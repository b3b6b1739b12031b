"""The tree checker used by the GPU parity tests, tested on the CPU: it must
accept the oracle's own tree, reject host-side perturbed copies of it (a
changed parent, token, depth or score), and excuse a mismatch only at an
oracle near tie or at a candidate set that really differs at a near tie."""
import copy

import numpy as np
import pytest

import oracle.domino_oracle as O
from draft_head_gb300 import synth
from tests.tree_check import NEAR_TIE, compare_tree, compare_trees


def _oracle_tree():
    cfg = dict(index=98, dtype="f32", d=16, V=40, g=8, e=16, r=8, block=6, batch=3, temperature=0.0)
    case = synth.make_case(cfg, 17, strong_coupling=True)
    case["w_lm"] = (case["w_lm"] * 6.0).astype(np.float32)  # peaked: deeper trees
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    N, M = 12, 4
    o = O.tree_build(head, case["H"], L, case["anchor"], N, M)
    g = tuple(o[k].astype(np.int32) for k in ("node_token", "node_parent", "node_depth")) + (
        o["node_score"].astype(np.float32),)
    return o, g, N


def _copy(g):
    return tuple(x.copy() for x in g)


def _clear_node(o, N):
    """(request, node) pairs whose pop is not a near tie and where no
    candidate boundary is a near tie: a mismatch there must fail."""
    out = []
    for b in range(o["node_token"].shape[0]):
        if np.min(o["cand_gap"][b]) < NEAR_TIE:
            continue
        for k in range(2, N + 1):
            if o["pop_margin"][b, k] >= NEAR_TIE and o["node_token"][b, k] >= 0:
                out.append((b, k))
    return out


def test_checker_accepts_the_oracle_tree():
    o, g, N = _oracle_tree()
    assert compare_trees(g, o, N, range(3)) == (3, 0)
    assert np.max(o["node_depth"]) >= 2  # the perturbations below reach below the root's children


@pytest.mark.parametrize("field", ["parent", "token", "depth", "score"])
def test_checker_rejects_a_perturbed_tree(field):
    o, g, N = _oracle_tree()
    nodes = _clear_node(o, N)
    assert nodes, "the fixture needs a node with a clear pop margin"
    for b, k in nodes[:4]:
        bad = _copy(g)
        tok, par, dep, sco = bad
        if field == "parent":
            par[b, k] = (par[b, k] + 1) % k  # another earlier node
        elif field == "token":
            tok[b, k] = tok[b, k] + 1
        elif field == "depth":
            dep[b, k] = dep[b, k] + 1
        else:
            sco[b, k] = sco[b, k] - 0.01
        with pytest.raises(AssertionError):
            compare_tree(bad, o, b, N)


def test_checker_excuses_an_oracle_pop_near_tie_only_there():
    o, g, N = _oracle_tree()
    b, k = _clear_node(o, N)[0]
    bad = _copy(g)
    bad[0][b, k] += 1
    o2 = copy.deepcopy(o)
    o2["pop_margin"][b, k] = 0.5 * NEAR_TIE
    assert compare_tree(bad, o2, b, N) == "near_tie"
    # A near tie at another pop does not excuse this one.
    o3 = copy.deepcopy(o)
    o3["pop_margin"][b, k - 1] = 0.0
    with pytest.raises(AssertionError):
        compare_tree(bad, o3, b, N)


def test_checker_excuses_a_candidate_set_difference_only_at_a_near_tie():
    o, g, N = _oracle_tree()
    b, k = _clear_node(o, N)[0]
    t = int(o["node_depth"][b, k]) - 1  # the set node k was drawn from
    bad = _copy(g)
    bad[0][b, k] += 1
    gpu_cands = o["cands"].copy()
    gpu_cands[b, t, -1] = 10_000 + gpu_cands[b, t, -1]  # the GPU kept another M-th candidate
    o2 = copy.deepcopy(o)
    o2["cand_gap"][b, t] = 0.5 * NEAR_TIE
    assert compare_tree(bad, o2, b, N, gpu_cands=gpu_cands) == "near_tie"
    # The same set difference at a clear boundary is a GPU error, not a tie.
    with pytest.raises(AssertionError):
        compare_tree(bad, o, b, N, gpu_cands=gpu_cands)
    # A near-tie boundary whose sets agree excuses nothing.
    with pytest.raises(AssertionError):
        compare_tree(bad, o2, b, N, gpu_cands=o["cands"])
    # Nor does a set difference at a depth that neither mismatching node
    # draws from (the children of node k's depth).
    assert t + 1 < o["cands"].shape[1]
    gc2 = o["cands"].copy()
    gc2[b, t + 1, -1] += 10_000
    o3 = copy.deepcopy(o)
    o3["cand_gap"][b, t + 1] = 0.0
    with pytest.raises(AssertionError):
        compare_tree(bad, o3, b, N, gpu_cands=gc2)
