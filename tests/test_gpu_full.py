"""Full-size parity on the Qwen3-shaped workloads (vocabulary 151936, GRU 1024,
rank 256, block 16), in the launch configuration the benchmark times. The
oracle recomputes sampled base-logit entries one by one and whole chains /
trees for sampled requests."""
import numpy as np
import pytest
import torch

import oracle.domino_oracle as O
from draft_head_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if torch.cuda.is_available():
    from draft_head_gb300 import binding as B
    from tests import parity_log
    from tests.gpu_harness import (GpuCase, NEAR_TIE, TOL, check_logits, compare_forced, compare_tokens,
                                   compare_trees, gpu_candidates, to_dev)


def _case(name, **kw):
    return synth.make_case(synth.CONFIGS[name], synth.case_seed(name, 0), **kw)


def _oracle_subset(case, reqs, temperature=0.0, force=None):
    head = O.prepare_head(case)
    bs, P, V = case["batch"], case["P"], case["V"]
    L = np.full((bs, P, V), np.nan)
    L[reqs] = O.base_logits(case["H"][reqs], case["w_lm"])
    G = case["gumbel"][:, 1:, :] if temperature > 0.0 else None
    toks, margins, logits = O.draft_chain(head, case["H"], L, case["anchor"], temperature=temperature,
                                          gumbel=G, force=force, want_logits=force is not None,
                                          requests=reqs)
    return head, L, toks, margins, logits


def _check_base(case, gc, L, Ph, n_samples=3000):
    rng = np.random.default_rng(1)
    rows = rng.integers(0, case["batch"] * case["P"], size=n_samples)
    cols = rng.integers(0, case["V"], size=n_samples)
    cols[:8] = [0, 1, 127, 128, case["V"] - 129, case["V"] - 128, case["V"] - 2, case["V"] - 1]
    ref = O.base_logit_entries(case["H"], case["w_lm"], rows, cols)
    got = L.view(-1, case["V"]).cpu().numpy()[rows, cols]
    assert np.max(np.abs(got - ref)) < 1e-3
    refp = O.widen(case["H"]).reshape(-1, case["d"]) @ O.widen(case["w1"])[:, :case["d"]].T
    assert np.max(np.abs(Ph.view(-1, case["r"]).cpu().numpy() - refp)) < 1e-3


def test_qwen3_4b_bs1_greedy_chain_and_verify():
    case = _case("qwen3_4b_bs1")
    gc = GpuCase(case)
    L, Ph = gc.base()
    _check_base(case, gc, L, Ph)
    _, Lo, toks, margins, _ = _oracle_subset(case, [0])
    gt, _ = gc.chain(L, Ph)
    compared, ties = compare_tokens(gt.cpu().numpy(), toks, margins)
    print(f"qwen3_4b_bs1: {compared} tokens bit-exact, {ties} near-tie divergences")
    gf, glo = gc.chain(L, Ph, force=toks, want_logits=True)
    _, _, tf, mf, lf = _oracle_subset(case, [0], force=toks)
    check_logits(glo.cpu().numpy(), lf, "bf16")
    compare_forced(gf.cpu().numpy(), tf, mf)
    # Verification against targets that flip each oracle draft token w.p. 0.2.
    tgt = synth.make_targets(toks, "flip", 0.2, case["V"], seed=case["seed"])
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    adv = torch.empty(1, dtype=torch.int32, device="cuda")
    B.domino_verify(gt, to_dev(tgt), 1, case["P"], acc, adv)
    ra, rv = O.verify(toks, tgt)
    if ties == 0:
        assert acc.item() == ra[0] and adv.item() == rv[0]
    assert gc.status() == 0


def test_qwen3_4b_bs64_gumbel_chain():
    case = _case("qwen3_4b_bs64")
    gc = GpuCase(case)
    L, Ph = gc.base()
    _check_base(case, gc, L, Ph)
    reqs = [0, 37, 63]
    _, _, toks, margins, _ = _oracle_subset(case, reqs, temperature=1.0)
    gt, _ = gc.chain(L, Ph, temperature=1.0)
    compare_tokens(gt.cpu().numpy(), toks, margins, requests=reqs)
    force = np.where(toks >= 0, toks, 0)
    gf, glo = gc.chain(L, Ph, temperature=1.0, force=force, want_logits=True)
    _, _, tf, mf, lf = _oracle_subset(case, reqs, temperature=1.0, force=force)
    check_logits(glo.cpu().numpy()[reqs], lf[reqs], "bf16")
    compare_forced(gf.cpu().numpy(), tf, mf, requests=reqs)
    assert gc.status() == 0


def test_qwen3_8b_bs32_chain_and_verify():
    case = _case("qwen3_8b_bs32")
    gc = GpuCase(case)
    L, Ph = gc.base()
    _check_base(case, gc, L, Ph, n_samples=1500)
    reqs = [0, 31]
    _, _, toks, margins, _ = _oracle_subset(case, reqs)
    gt, _ = gc.chain(L, Ph)
    _, ties = compare_tokens(gt.cpu().numpy(), toks, margins, requests=reqs)
    tgt = synth.make_targets(np.where(toks >= 0, toks, 0), "match", 0.85, case["V"], seed=case["seed"])
    acc = torch.empty(case["batch"], dtype=torch.int32, device="cuda")
    adv = torch.empty_like(acc)
    B.domino_verify(gt, to_dev(tgt), case["batch"], case["P"], acc, adv)
    ra, rv = O.verify(np.where(toks >= 0, toks, 0), tgt)
    if ties == 0:
        assert np.array_equal(acc.cpu().numpy()[reqs], ra[reqs])
        assert np.array_equal(adv.cpu().numpy()[reqs], rv[reqs])
    assert gc.status() == 0


@pytest.mark.parametrize("T", [0.0, 0.5])
def test_qwen3_4b_tree_bs16(T):
    """The tree workload (batch 16, N = 16, M = 64) at the greedy setting and
    at decoding temperature 0.5: every request compared with the oracle under
    the strict rule (a mismatch only at an oracle near tie or at a candidate
    set that really differs at a near tie)."""
    case = _case("qwen3_4b_tree")
    N, M = 16, 64
    gc = GpuCase(case, n_nodes=N, top_m=M)
    L, Ph = gc.base()
    bs = case["batch"]
    tok = torch.empty(bs, N + 1, dtype=torch.int32, device="cuda")
    par, dep = torch.empty_like(tok), torch.empty_like(tok)
    sco = torch.empty(bs, N + 1, dtype=torch.float32, device="cuda")
    B.dominotree_build(gc.head, L, Ph, gc.anchor, bs, case["P"], N, M, tok, par, dep, sco, gc.ws, temperature=T)
    head = O.prepare_head(case)
    Lo = O.base_logits(case["H"], case["w_lm"])
    o = O.tree_build(head, case["H"], Lo, case["anchor"], N, M, temperature=T)
    g = (tok.cpu().numpy(), par.cpu().numpy(), dep.cpu().numpy(), sco.cpu().numpy())
    exact, ties = compare_trees(g, o, N, range(bs), gpu_cands=gpu_candidates(L, M))
    parity_log.trees(exact, ties)
    near = int(np.sum(np.min(o["cand_gap"], axis=1) < NEAR_TIE))
    print(f"qwen3_4b_tree T={T}: {exact} of {bs} trees bit-exact, {ties} up to a near tie; "
          f"{near} requests have a top-M boundary gap below 1e-3")
    assert ties == 0
    # Structural invariants for every request.
    gt, gp, gd, gs = g
    for b in range(bs):
        assert np.all(gt[b, 1:] >= 0)
        for k in range(1, N + 1):
            assert 0 <= gp[b, k] < k and gd[b, k] == gd[b, gp[b, k]] + 1
            assert gs[b, k] <= gs[b, gp[b, k]]
    assert gc.status() == 0


def test_qwen3_4b_bs3_gumbel_small_batch_chain():
    """Batch 3 with sampling at full vocabulary: the small-batch chain kernel's
    three row stores (tensor memory, shared memory, streamed) are all in use."""
    cfg = dict(synth.CONFIGS["qwen3_4b_bs1"], batch=3, temperature=1.0)
    case = synth.make_case(cfg, 4242)
    gc = GpuCase(case)
    L, Ph = gc.base()
    reqs = [0, 2]
    _, _, toks, margins, _ = _oracle_subset(case, reqs, temperature=1.0)
    gt, _ = gc.chain(L, Ph, temperature=1.0)
    compare_tokens(gt.cpu().numpy(), toks, margins, requests=reqs)
    force = np.where(toks >= 0, toks, 0)
    gf, glo = gc.chain(L, Ph, temperature=1.0, force=force, want_logits=True)
    _, _, tf, mf, lf = _oracle_subset(case, reqs, temperature=1.0, force=force)
    check_logits(glo.cpu().numpy()[reqs], lf[reqs], "bf16")
    compare_forced(gf.cpu().numpy(), tf, mf, requests=reqs)
    assert gc.status() == 0


def test_full_size_headoff_chain_marginal_tree_and_tree_verify():
    """The head-off baselines and tree acceptance at the Qwen3 vocabulary: the
    batch-64 Gumbel head-off chain on sampled rows, the batch-16 marginal tree
    (N = 16, M = 64) on sampled requests, and the acceptance walk of that tree."""
    V, P = 151936, 15
    # Head-off chain, batch 64, T = 1.
    bs = 64
    L = synth.normal((bs, P, V), 1.0, 9101, 0)
    g_full = synth.gumbel_noise((bs, P + 1, V), 9101)
    Ld, gd = to_dev(L), to_dev(g_full)
    toks = torch.empty(bs, P, dtype=torch.int32, device="cuda")
    ws = B.workspace(B.domino_headoff_workspace_bytes(bs, P, V))
    B.domino_draft_chain_headoff(Ld, bs, P, V, 1.0, gd[:, 1:, :], (P + 1) * V, toks, ws)
    got = toks.cpu().numpy()
    assert B.domino_last_status(ws) == 0
    reqs = [0, 17, 63]
    ot, om = O.draft_chain_headoff(L[reqs].astype(np.float64), 1.0, g_full[reqs, 1:, :])
    bad = (got[reqs] != ot) & ~(om < NEAR_TIE)
    assert not bad.any()
    del Ld, gd, L, g_full
    # Marginal tree, batch 16, N = 16, M = 64, and its acceptance.
    bs, N, M = 16, 16, 64
    L = synth.normal((bs, P, V), 1.0, 9102, 0)
    anchor = (np.arange(bs, dtype=np.int32) * 977) % V
    shape = (bs, N + 1)
    out = [torch.empty(shape, dtype=torch.int32, device="cuda") for _ in range(3)]
    sc = torch.empty(shape, dtype=torch.float32, device="cuda")
    ws = B.workspace(B.domino_headoff_workspace_bytes(bs, P, V, N, M))
    B.dominotree_build_marginal(to_dev(L), to_dev(anchor), bs, P, V, N, M, out[0], out[1], out[2], sc, ws)
    g = tuple(x.cpu().numpy() for x in out) + (sc.cpu().numpy(),)
    assert B.domino_last_status(ws) == 0
    # Every request under the strict rule.
    o_all = O.tree_build_marginal(L.astype(np.float64), anchor, N, M)
    exact, ties = compare_trees(g, o_all, N, range(bs), gpu_cands=gpu_candidates(to_dev(L), M))
    parity_log.trees(exact, ties)
    assert ties == 0
    sel = [0, 7, 15]
    o = {k: v[sel] for k, v in o_all.items()}
    tok = o["node_token"].astype(np.int32)
    par = o["node_parent"].astype(np.int32)
    tgt = synth.make_tree_targets(tok, par, 0.2, V, seed=9102)
    acc = torch.empty(len(sel), dtype=torch.int32, device="cuda")
    adv = torch.empty_like(acc)
    path = torch.empty(len(sel), N + 1, dtype=torch.int32, device="cuda")
    mask = torch.empty(len(sel), N + 1, N + 1, dtype=torch.uint8, device="cuda")
    B.dominotree_verify(to_dev(tok), to_dev(par), to_dev(tgt), len(sel), N, acc, adv, path, mask)
    oa, oad, op, om2 = O.tree_verify(tok, par, tgt)
    assert np.array_equal(acc.cpu().numpy(), oa) and np.array_equal(adv.cpu().numpy(), oad)
    assert np.array_equal(path.cpu().numpy(), op) and np.array_equal(mask.cpu().numpy(), om2)
