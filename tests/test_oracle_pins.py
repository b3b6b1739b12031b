"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- hand-worked values, closed forms, library routines (torch, scipy),
brute-force enumeration on tiny inputs, and invariants the method implies.
CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.domino_oracle as O
from draft_head_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def tiny_case(seed=7, strong=False, w2_zero=False, batch=1, gumbel=False, **over):
    cfg = dict(synth.CONFIGS["tiny_f32"])
    cfg.update(over)
    return synth.make_case(cfg, seed, strong_coupling=strong, w2_zero=w2_zero, batch=batch,
                           gumbel=gumbel)


def micro_cfg(**over):
    c = dict(index=99, dtype="f32", d=8, V=12, g=4, e=8, r=4, block=4, batch=1,
             temperature=0.0)
    c.update(over)
    return c


# --------------------------------------------------------------------------- P1
def test_param_count_matches_quoted_head_size():
    gs = _load("head_shapes.json")
    n8 = O.head_param_count(gs["qwen3_8b_hidden"], gs["qwen3_8b_hidden"], gs["gru_hidden"],
                            gs["rank"], gs["vocab"])
    assert n8 == 38_895_616 + 1_310_720 + 15_728_640 + 6_144
    assert abs(n8 / 1e6 - gs["quoted_params_millions"]) <= gs["quoted_rounding_millions"]
    # A separately trained embedding table would not match the quoted figure.
    n8_own = O.head_param_count(4096, 4096, 1024, 256, 151936, shared_embedding=False)
    assert abs(n8_own / 1e6 - gs["quoted_params_millions"]) > 100


# --------------------------------------------------------------------------- P2
@pytest.mark.parametrize("idx", [0, 1, 2])
def test_gru_hand_worked(idx):
    c = _load("gru_hand.json")["cases"][idx]
    got = O.gru_cell(np.array(c["x"], float), np.array(c["h"], float),
                     np.array(c["w_ih"], float), np.array(c["w_hh"], float),
                     np.array(c["b_ih"], float), np.array(c["b_hh"], float))
    np.testing.assert_allclose(got, c["expected"], rtol=0, atol=1e-15)


def test_gru_matches_torch_grucell():
    rng = np.random.default_rng(3)
    e, g = 6, 5
    cell = torch.nn.GRUCell(e, g).double()
    with torch.no_grad():
        for p in cell.parameters():
            p.copy_(torch.from_numpy(rng.normal(0, 0.7, size=tuple(p.shape))))
    x = rng.normal(size=e)
    h = rng.uniform(-0.9, 0.9, size=g)
    ref = cell(torch.from_numpy(x)[None], torch.from_numpy(h)[None])[0].detach().numpy()
    got = O.gru_cell(x, h, cell.weight_ih.detach().numpy(), cell.weight_hh.detach().numpy(),
                     cell.bias_ih.detach().numpy(), cell.bias_hh.detach().numpy())
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_silu_closed_forms_and_torch():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(O.silu(-1.0) - (-1.0 / (1.0 + math.e))) < 1e-16
    t = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(O.silu(t), torch.nn.functional.silu(torch.from_numpy(t)).numpy(),
                               rtol=1e-14, atol=1e-300)


# --------------------------------------------------------------------------- P5
def test_base_logits_brute_force():
    rng = np.random.default_rng(0)
    H = rng.normal(size=(2, 3, 5)).astype(np.float32)
    W = rng.normal(size=(7, 5)).astype(np.float32)
    got = O.base_logits(H, W)
    for b, i, v in itertools.product(range(2), range(3), range(7)):
        s = 0.0
        for k in range(5):
            s += float(H[b, i, k]) * float(W[v, k])
        assert abs(got[b, i, v] - s) < 1e-12
    ent = O.base_logit_entries(H, W, [0, 5], [6, 2])
    assert abs(ent[0] - got[0, 0, 6]) < 1e-12 and abs(ent[1] - got[1, 2, 2]) < 1e-12


def test_base_logits_bf16_widening_is_exact():
    x = np.array([1.0, -2.5, 3.140625, 1e-3], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(x)
    w = O.widen(bits)
    assert w[0] == 1.0 and w[1] == -2.5 and w[2] == 3.140625
    # 1e-3 = 0x3A83126F in fp32; the dropped half 0x126F < 0x8000 rounds down.
    assert bits[3] == 0x3A83 and w[3] == 0.00099945068359375
    # Ties go to even: 0x3F808000 (1.00390625) -> 0x3F80, 0x3F818000 -> 0x3F82.
    t = np.array([1.00390625, 1.01171875], dtype=np.float32)
    assert list(synth.f32_to_bf16_bits(t)) == [0x3F80, 0x3F82]


# --------------------------------------------------------------------------- P3
def test_argmax_ties_to_lowest_id():
    v = np.array([0.5, 2.0, -1.0, 2.0, 2.0])
    assert O._fp32_argmax(v)[0] == 1
    rng = np.random.default_rng(1)
    for _ in range(200):
        x = rng.integers(-3, 4, size=17).astype(float)  # many exact ties
        best = O._fp32_argmax(x)[0]
        assert x[best] == x.max() and all(x[j] < x.max() for j in range(best))


def test_argmax_decides_in_fp32():
    # Two fp64 values that round to the same fp32 value tie in fp32 -> lowest id.
    a = 1.0
    b = 1.0 + 2.0 ** -30
    assert O._fp32_argmax(np.array([a, b]))[0] == 0


# --------------------------------------------------------------------------- chain
def _torch_chain(case, force=None, want_u=False):
    """Independent chain built from library routines: torch.nn.GRUCell, F.silu, matmul."""
    f = lambda k: torch.from_numpy(O.widen(case[k]))
    g, e = case["g"], case["e"]
    cell = torch.nn.GRUCell(e, g).double()
    with torch.no_grad():
        cell.weight_ih.copy_(f("w_ih")); cell.weight_hh.copy_(f("w_hh"))
        cell.bias_ih.copy_(f("b_ih")); cell.bias_hh.copy_(f("b_hh"))
    H, Wlm, emb, W1, W2 = f("H"), f("w_lm"), f("emb"), f("w1"), f("w2")
    bs, P = H.shape[0], H.shape[1]
    toks = np.zeros((bs, P), np.int64)
    logits = np.zeros((bs, P, case["V"]))
    us = np.zeros((bs, P, case["r"]))
    with torch.no_grad():
        for b in range(bs):
            h = cell(emb[int(case["anchor"][b])][None], torch.zeros(1, g, dtype=torch.float64))
            for i in range(P):
                u = torch.nn.functional.silu(W1 @ torch.cat([H[b, i], h[0]]))
                L = Wlm @ H[b, i] + W2 @ u
                logits[b, i] = L.numpy()
                us[b, i] = u.numpy()
                toks[b, i] = int(torch.argmax(L.float()))
                nxt = toks[b, i] if force is None else force[b, i]
                h = cell(emb[int(nxt)][None], h)
    if want_u:
        return toks, logits, us
    return toks, logits


@pytest.mark.parametrize("strong", [False, True])
def test_chain_matches_library_built_chain(strong):
    case = tiny_case(seed=11, strong=strong, batch=2)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    toks, margins, logits = O.draft_chain(head, case["H"], L, case["anchor"], want_logits=True)
    rt, rl = _torch_chain(case)
    np.testing.assert_allclose(logits, rl, rtol=0, atol=1e-11)
    ok = margins > 1e-9
    assert np.array_equal(toks[ok], rt[ok])


def test_chain_w2_zero_is_parallel_draft():
    case = tiny_case(seed=5, w2_zero=True, batch=3)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    toks, _, logits = O.draft_chain(head, case["H"], L, case["anchor"], want_logits=True)
    assert np.array_equal(logits, L)  # bit for bit: the correction is exactly zero
    assert np.array_equal(toks, np.argmax(L.astype(np.float32), axis=-1))


def test_chain_forced_with_own_draft_is_identical():
    case = tiny_case(seed=9, strong=True, batch=2)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    t1, _, l1 = O.draft_chain(head, case["H"], L, case["anchor"], want_logits=True)
    t2, _, l2 = O.draft_chain(head, case["H"], L, case["anchor"], force=t1, want_logits=True)
    assert np.array_equal(t1, t2) and np.array_equal(l1, l2)


def test_chain_causality_and_indexing():
    """Position i depends on H_i, the anchor and the GRU inputs before it only."""
    case = tiny_case(seed=13, strong=True)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    P = case["P"]
    f0 = np.zeros((1, P), np.int64)
    f1 = f0.copy(); f1[0, 1] = 17
    _, _, la = O.draft_chain(head, case["H"], L, case["anchor"], force=f0, want_logits=True)
    _, _, lb = O.draft_chain(head, case["H"], L, case["anchor"], force=f1, want_logits=True)
    assert np.array_equal(la[0, :2], lb[0, :2])          # positions 0, 1 unaffected
    assert np.max(np.abs(la[0, 2] - lb[0, 2])) > 1e-6    # position 2 sees the changed token
    # H_i enters position i only (through L_base and through [H_i; S]).
    H2 = case["H"].copy(); H2[0, 1] += 1.0
    _, _, lc = O.draft_chain(head, H2, L, case["anchor"], force=f0, want_logits=True)
    assert np.array_equal(la[0, 0], lc[0, 0]) and np.array_equal(la[0, 2], lc[0, 2])
    assert np.max(np.abs(la[0, 1] - lc[0, 1])) > 1e-6
    # The anchor drives the first state: a different anchor changes position 0.
    _, _, ld = O.draft_chain(head, case["H"], L, (case["anchor"] + 1) % case["V"], force=f0,
                             want_logits=True)
    assert np.max(np.abs(la[0, 0] - ld[0, 0])) > 1e-6


def test_chain_gumbel_max():
    case = tiny_case(seed=21, batch=2, gumbel=True)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    G = case["gumbel"][:, 1:, :]
    zero = np.zeros_like(G)
    tg, _, _ = O.draft_chain(head, case["H"], L, case["anchor"])
    tz, _, _ = O.draft_chain(head, case["H"], L, case["anchor"], temperature=1.0, gumbel=zero)
    assert np.array_equal(tg, tz)  # zero noise at T=1 is greedy
    big = zero.copy(); big[:, :, 123] = 1e6
    tb, _, _ = O.draft_chain(head, case["H"], L, case["anchor"], temperature=1.0, gumbel=big)
    assert np.all(tb == 123)
    # Temperature scales the logits before the noise is added.
    t1, _, lg = O.draft_chain(head, case["H"], L, case["anchor"], temperature=0.5, gumbel=G,
                              want_logits=True)
    assert np.array_equal(t1, np.argmax((lg / 0.5 + G).astype(np.float32), axis=-1))


@pytest.mark.parametrize("T", [0.0, 0.7])
def test_chain_stats_match_library_built_chain(T):
    """Reading S6: u_i is the library-built chain's SiLU(W1 [H_i; S]) and lse_i
    is scipy's logsumexp of its logits / T' (T' = 1 at T = 0); the tokens are
    the chain's own."""
    from scipy.special import logsumexp
    case = tiny_case(seed=23, strong=True, batch=2, gumbel=True)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    G = case["gumbel"][:, 1:, :]
    toks, _, us, lse = O.draft_chain_stats(head, case["H"], L, case["anchor"], temperature=T, gumbel=G)
    want_toks, _, _ = O.draft_chain(head, case["H"], L, case["anchor"], temperature=T, gumbel=G)
    assert np.array_equal(toks, want_toks)
    # Teacher-force the library chain with the drafted tokens so both see the same GRU inputs.
    _, rl, ru = _torch_chain(case, force=toks, want_u=True)
    np.testing.assert_allclose(us, ru, rtol=0, atol=1e-12)
    tau = T if T > 0 else 1.0
    np.testing.assert_allclose(lse, logsumexp(rl / tau, axis=-1), rtol=0, atol=1e-10)


def test_chain_stats_closed_form():
    """W2 = 0 and a constant base row c: lse = c / T + log V; u still follows
    the GRU (nonzero)."""
    case = tiny_case(seed=3, w2_zero=True, batch=1)
    head = O.prepare_head(case)
    V, P = case["V"], case["P"]
    L = np.full((1, P, V), 2.5)
    _, _, us, lse = O.draft_chain_stats(head, case["H"], L, case["anchor"], temperature=0.5,
                                        gumbel=np.zeros((1, P, V)))
    np.testing.assert_allclose(lse, 2.5 / 0.5 + math.log(V), rtol=0, atol=1e-12)
    assert np.all(np.abs(us) > 0)


def test_gumbel_noise_distribution():
    g = synth.gumbel_noise((200000,), seed=4).astype(np.float64)
    assert abs(g.mean() - 0.5772156649) < 0.01           # Euler-Mascheroni constant
    assert abs(g.var() - math.pi ** 2 / 6) < 0.03


# --------------------------------------------------------------------------- P6
def test_verify_brute_force_and_closed_forms():
    rng = np.random.default_rng(2)
    d = rng.integers(0, 3, size=(500, 6))
    t = rng.integers(0, 3, size=(500, 6))
    acc, adv = O.verify(d, t)
    for b in range(500):
        k = max(k for k in range(7) if np.array_equal(d[b, :k], t[b, :k]))
        assert acc[b] == k and adv[b] == k + 1
    same = rng.integers(0, 9, size=(4, 15))
    a2, v2 = O.verify(same, same)
    assert np.all(a2 == 15) and np.all(v2 == 16)
    t3 = same.copy(); t3[:, 0] += 1
    a3, v3 = O.verify(same, t3)
    assert np.all(a3 == 0) and np.all(v3 == 1)


@pytest.mark.parametrize("mode,p,expect", [("flip", 0.2, None), ("match", 0.85, None)])
def test_verify_expected_accept_length(mode, p, expect):
    P, n = 15, 40000
    keep = (1 - p) if mode == "flip" else p
    closed = sum(keep ** k for k in range(1, P + 1))  # E[accept] = sum_k p^k
    draft = np.random.default_rng(8).integers(0, 1000, size=(n, P))
    target = synth.make_targets(draft, mode, p, 1000, seed=5)
    acc, _ = O.verify(draft, target)
    sd = acc.std() / math.sqrt(n)
    assert abs(acc.mean() - closed) < 4 * sd
    if mode == "flip":
        assert abs(closed - 3.859) < 1e-3
    else:
        assert abs(closed - 5.1717) < 1e-3


# --------------------------------------------------------------------------- top-M
def test_top_m_matches_stable_sort():
    rng = np.random.default_rng(4)
    for _ in range(50):
        x = rng.integers(-5, 6, size=300).astype(np.float64) * 0.25  # heavy ties
        ids, gap = O.top_m(x, 64)
        ref = np.argsort(-x, kind="stable")[:64]
        assert np.array_equal(ids, ref)
        assert gap == x[ref[63]] - x[np.argsort(-x, kind="stable")[64]]


def test_logsumexp_matches_scipy():
    from scipy.special import logsumexp
    x = np.random.default_rng(0).normal(size=64) * 10
    assert abs(O._logsumexp(x) - logsumexp(x)) < 1e-12


# --------------------------------------------------------------------------- tree
def _torch_scores_all_paths(case, L, M, P, tau=None):
    """Every node of the full candidate tree (depth <= P), scored by an
    independent library-built chain: torch GRUCell, F.silu, torch.logsumexp
    (tau given: F.log_softmax of the logits divided by tau)."""
    f = lambda k: torch.from_numpy(O.widen(case[k]))
    g, e = case["g"], case["e"]
    cell = torch.nn.GRUCell(e, g).double()
    with torch.no_grad():
        cell.weight_ih.copy_(f("w_ih")); cell.weight_hh.copy_(f("w_hh"))
        cell.bias_ih.copy_(f("b_ih")); cell.bias_hh.copy_(f("b_hh"))
    H, emb, W1, W2 = f("H"), f("emb"), f("w1"), f("w2")
    Lt = torch.from_numpy(L)
    cands = [torch.from_numpy(np.argsort(-L[0, t].astype(np.float32), kind="stable")[:M])
             for t in range(P)]
    out = {}
    with torch.no_grad():
        def rec(path, h, score):
            t = len(path)
            if t == P:
                return
            u = torch.nn.functional.silu(W1 @ torch.cat([H[0, t], h[0]]))
            C = cands[t]
            l = Lt[0, t, C] + W2[C] @ u
            lp = l - torch.logsumexp(l, 0) if tau is None else torch.nn.functional.log_softmax(l / tau, 0)
            for c, v in zip(C.tolist(), lp.tolist()):
                p2 = path + (c,)
                out[p2] = score + v
                rec(p2, cell(emb[c][None], h), score + v)
        rec((), cell(emb[int(case["anchor"][0])][None], torch.zeros(1, g, dtype=torch.float64)), 0.0)
    return out


def _oracle_paths(tr, b=0):
    tok, par = tr["node_token"][b], tr["node_parent"][b]
    paths = {}
    for k in range(1, len(tok)):
        if tok[k] < 0:
            continue
        p = par[k]
        paths[k] = (paths[p] if p > 0 else ()) + (int(tok[k]),)
    return paths


@pytest.mark.parametrize("seed,strong", [(1, True), (2, True), (3, False)])
def test_tree_equals_brute_force_top_n(seed, strong):
    cfg = micro_cfg()
    case = synth.make_case(cfg, seed, strong_coupling=strong)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    P, M, N = case["P"], 3, 10
    allp = _torch_scores_all_paths(case, L, M, P)
    assert len(allp) == 3 + 9 + 27
    tr = O.tree_build(head, case["H"], L, case["anchor"], N, M)
    paths = _oracle_paths(tr)
    best = sorted(allp.items(), key=lambda kv: -kv[1])[:N]
    assert [p for p, _ in best] == [paths[k] for k in range(1, N + 1)]  # same nodes, pop order
    for k in range(1, N + 1):
        assert abs(tr["node_score"][0, k] - allp[paths[k]]) < 1e-5


@pytest.mark.parametrize("seed,T", [(1, 0.5), (2, 0.5), (11, 2.0)])
def test_tempered_tree_equals_brute_force_top_n(seed, T):
    """Reading T10 at T > 0: the best-first tree is the N best nodes of the full
    candidate tree scored by log-softmax(l / T) over each slice."""
    cfg = micro_cfg()
    case = synth.make_case(cfg, seed, strong_coupling=True)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    P, M, N = case["P"], 3, 10
    allp = _torch_scores_all_paths(case, L, M, P, tau=T)
    tr = O.tree_build(head, case["H"], L, case["anchor"], N, M, temperature=T)
    paths = _oracle_paths(tr)
    best = sorted(allp.items(), key=lambda kv: -kv[1])[:N]
    assert [p for p, _ in best] == [paths[k] for k in range(1, N + 1)]
    for k in range(1, N + 1):
        assert abs(tr["node_score"][0, k] - allp[paths[k]]) < 1e-5
    # Greedy decoding (T = 0) ranks by the untempered log-softmax: the T = 1 tree.
    t0 = O.tree_build(head, case["H"], L, case["anchor"], N, M, temperature=0.0)
    t1 = O.tree_build(head, case["H"], L, case["anchor"], N, M, temperature=1.0)
    for key in ("node_token", "node_parent", "node_depth", "node_score"):
        assert np.array_equal(t0[key], t1[key])


def test_tempered_tree_is_the_tree_of_scaled_logits():
    """Dividing every logit by T = 1/2 is the same as doubling W_lm and W2 at
    T = 1 (exact in binary floating point): the same tree, score for score. A
    temperature applied to only one of the two logit terms fails this."""
    cfg = micro_cfg(block=5)
    case = synth.make_case(cfg, 12, strong_coupling=True, batch=2)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    a = O.tree_build(head, case["H"], L, case["anchor"], 14, 4, temperature=0.5)
    c2 = dict(case, w_lm=case["w_lm"] * np.float32(2.0), w2=case["w2"] * np.float32(2.0))
    h2 = O.prepare_head(c2)
    L2 = O.base_logits(c2["H"], c2["w_lm"])
    assert np.array_equal(L2, 2.0 * L)
    b = O.tree_build(h2, c2["H"], L2, c2["anchor"], 14, 4, temperature=1.0)
    for key in ("node_token", "node_parent", "node_depth", "node_score", "cands"):
        assert np.array_equal(a[key], b[key])
    # ... and differs from the untempered tree on this case (the check has teeth).
    u = O.tree_build(head, case["H"], L, case["anchor"], 14, 4)
    assert not np.array_equal(u["node_score"], a["node_score"])
    # Marginal tree: the same identity with W_lm alone.
    m = O.tree_build_marginal(L, case["anchor"], 14, 4, temperature=0.5)
    m2 = O.tree_build_marginal(L2, case["anchor"], 14, 4)
    for key in ("node_token", "node_parent", "node_depth", "node_score"):
        assert np.array_equal(m[key], m2[key])


def test_tree_invariants_and_single_path():
    cfg = micro_cfg(block=5)
    case = synth.make_case(cfg, 4, strong_coupling=True, batch=2)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    P, M, N = case["P"], 4, 12
    tr = O.tree_build(head, case["H"], L, case["anchor"], N, M)
    for b in range(2):
        tok, par, dep, sco = (tr[k][b] for k in ("node_token", "node_parent", "node_depth", "node_score"))
        assert dep[0] == 0 and par[0] == -1 and sco[0] == 0.0
        assert np.all(tok[1:] >= 0)  # exactly N drafted nodes
        for k in range(1, N + 1):
            assert 0 <= par[k] < k and dep[k] == dep[par[k]] + 1 and dep[k] <= P
            cset, _ = O.top_m(L[b, dep[k] - 1], M)
            assert tok[k] in cset
            assert sco[k] <= sco[par[k]]
        assert np.all(np.diff(sco[1:].astype(np.float64)) <= 0)  # pops never increase
    # M = 1: a single path of per-depth base argmax tokens, then the heap runs dry.
    tr1 = O.tree_build(head, case["H"], L, case["anchor"], 16, 1)
    for b in range(2):
        assert list(tr1["node_depth"][b, 1:P + 1]) == list(range(1, P + 1))
        assert list(tr1["node_parent"][b, 1:P + 1]) == list(range(0, P))
        assert np.array_equal(tr1["node_token"][b, 1:P + 1], np.argmax(L[b].astype(np.float32), -1))
        assert np.all(tr1["node_token"][b, P + 1:] == -1)


def test_tree_w2_zero_is_factorised():
    """W2 = 0: scores are sums of per-depth marginal log-probs over the M-slice."""
    cfg = micro_cfg()
    case = synth.make_case(cfg, 6, w2_zero=True)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    P, M, N = case["P"], 3, 9
    from scipy.special import logsumexp
    lp = []
    for t in range(P):
        C = np.argsort(-L[0, t].astype(np.float32), kind="stable")[:M]
        lp.append({int(c): L[0, t, c] - logsumexp(L[0, t, C]) for c in C})
    allp = {}
    for depth in range(1, P + 1):
        for path in itertools.product(*[list(lp[t].keys()) for t in range(depth)]):
            allp[path] = sum(lp[t][c] for t, c in enumerate(path))
    tr = O.tree_build(head, case["H"], L, case["anchor"], N, M)
    paths = _oracle_paths(tr)
    best = sorted(allp.items(), key=lambda kv: -kv[1])[:N]
    assert [p for p, _ in best] == [paths[k] for k in range(1, N + 1)]


# --------------------------------------------------------------------------- tree acceptance (f1)
def _golden(name):
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


@pytest.mark.parametrize("idx", range(3))
def test_tree_verify_hand_worked(idx):
    c = _golden("tree_verify_hand.json")["cases"][idx]
    acc, adv, path, mask = O.tree_verify([c["node_token"]], [c["node_parent"]], [c["target_next"]])
    assert acc[0] == c["accept"] and adv[0] == c["advanced"]
    assert list(path[0]) == c["path"]
    n1 = len(c["node_token"])
    want = np.zeros((n1, n1), dtype=np.uint8)
    for i, row in enumerate(c["mask_rows"]):
        want[i, row] = 1
    assert np.array_equal(mask[0], want)


def test_tree_verify_chain_shaped_tree_is_chain_verify():
    """A tree with one child per node is the chain: same accept lengths as verify()."""
    rng = np.random.default_rng(5)
    bs, P, V = 300, 7, 5
    draft = rng.integers(0, V, size=(bs, P))
    target = np.where(rng.random((bs, P)) < 0.7, draft, rng.integers(0, V, size=(bs, P)))
    tok = np.concatenate([np.full((bs, 1), 99), draft], 1)
    par = np.tile(np.arange(-1, P), (bs, 1))
    tnext = np.concatenate([target, rng.integers(0, V, size=(bs, 1))], 1)  # node i predicts position i
    acc, adv, path, _ = O.tree_verify(tok, par, tnext)
    acc2, adv2 = O.verify(draft, target)
    assert np.array_equal(acc, acc2) and np.array_equal(adv, adv2)
    for b in range(bs):
        assert list(path[b, :acc[b] + 1]) == list(range(acc[b] + 1))


def test_tree_verify_mask_is_transitive_closure_and_walk_is_valid():
    """Mask = reflexive-transitive closure of the parent relation, computed by
    boolean matrix powers; the accepted path follows target tokens."""
    cfg = micro_cfg(block=5)
    case = synth.make_case(cfg, 8, strong_coupling=True, batch=3)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    tr = O.tree_build(head, case["H"], L, case["anchor"], 12, 3)
    tgt = synth.make_tree_targets(tr["node_token"], tr["node_parent"], 0.3, cfg["V"], seed=8)
    acc, adv, path, mask = O.tree_verify(tr["node_token"], tr["node_parent"], tgt)
    n1 = tr["node_token"].shape[1]
    for b in range(3):
        A = np.zeros((n1, n1), dtype=np.int64)
        for i in range(1, n1):
            if tr["node_parent"][b, i] >= 0:
                A[i, tr["node_parent"][b, i]] = 1
        R = np.eye(n1, dtype=np.int64)
        Pw = np.eye(n1, dtype=np.int64)
        for _ in range(n1):
            Pw = np.minimum(Pw @ A, 1)
            R = np.maximum(R, Pw)
        assert np.array_equal(mask[b], R.astype(np.uint8))
        for k in range(1, acc[b] + 1):
            n, prev = path[b, k], path[b, k - 1]
            assert tr["node_parent"][b, n] == prev and tr["node_token"][b, n] == tgt[b, prev]
            assert tr["node_depth"][b, n] == k
        last = path[b, acc[b]]
        kids = [c for c in range(1, n1) if tr["node_parent"][b, c] == last and tr["node_token"][b, c] >= 0]
        assert all(tr["node_token"][b, c] != tgt[b, last] for c in kids)


# --------------------------------------------------------------------------- head-off baselines (f2)
@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_headoff_chain_is_w2_zero_chain(temperature):
    cfg = micro_cfg()
    case = synth.make_case(cfg, 9, w2_zero=True, batch=3, gumbel=temperature > 0)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    g = case["gumbel"][:, 1:, :] if temperature > 0 else None
    t_full, _, _ = O.draft_chain(head, case["H"], L, case["anchor"], temperature, g)
    t_off, _ = O.draft_chain_headoff(L, temperature, g)
    assert np.array_equal(t_full, t_off)
    dec = L if temperature == 0 else L / temperature + g
    assert np.array_equal(t_off, np.argmax(dec.astype(np.float32), -1))


def test_marginal_tree_is_w2_zero_tree_and_brute_force():
    cfg = micro_cfg()
    case = synth.make_case(cfg, 10, w2_zero=True)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    P, M, N = case["P"], 3, 9
    tm = O.tree_build_marginal(L, case["anchor"], N, M)
    tc = O.tree_build(head, case["H"], L, case["anchor"], N, M)
    for k in ("node_token", "node_parent", "node_depth", "node_score"):
        assert np.array_equal(tm[k], tc[k])
    from scipy.special import logsumexp
    lp = []
    for t in range(P):
        C = np.argsort(-L[0, t].astype(np.float32), kind="stable")[:M]
        lp.append({int(c): L[0, t, c] - logsumexp(L[0, t, C]) for c in C})
    allp = {}
    for depth in range(1, P + 1):
        for path in itertools.product(*[list(lp[t].keys()) for t in range(depth)]):
            allp[path] = sum(lp[t][c] for t, c in enumerate(path))
    paths = _oracle_paths(tm)
    best = sorted(allp.items(), key=lambda kv: -kv[1])[:N]
    assert [p for p, _ in best] == [paths[k] for k in range(1, N + 1)]


# --------------------------------------------------------------------------- verification at T > 0 (f3)
def _sample_from(probs, rng):
    return int(rng.choice(len(probs), p=probs))


def _stoch_case(rng, V, P, T, scale=1.0):
    L = rng.normal(0, scale, size=(1, P, V))
    Z = rng.normal(0, scale, size=(1, P + 1, V))
    q0 = np.exp(L[0, 0] / T) / np.exp(L[0, 0] / T).sum()
    return L, Z, q0


def test_stochastic_verify_is_lossless_first_token():
    """The first emitted token (the accepted draft token, or the residual draw
    at a rejection) is distributed as the target's p_0, whatever q_0 is."""
    rng = np.random.default_rng(11)
    V, P, T = 5, 2, 0.8
    L, Z, q0 = _stoch_case(rng, V, P, T)
    p0 = np.exp(Z[0, 0] / T) / np.exp(Z[0, 0] / T).sum()
    n = 40000
    counts = np.zeros(V)
    accepted0 = 0
    for _ in range(n):
        x = np.array([[_sample_from(q0, rng), _sample_from(q0, rng)]])
        u = rng.uniform(1e-7, 1 - 1e-7, size=(1, P))
        g = -np.log(-np.log(rng.uniform(1e-12, 1 - 1e-12, size=(1, V))))
        acc, _, nxt, _, _ = O.verify_stochastic(x, L, Z, u, g, T)
        first = x[0, 0] if acc[0] >= 1 else nxt[0]
        counts[first] += 1
        accepted0 += acc[0] >= 1
    sd = np.sqrt(n * p0 * (1 - p0))
    assert np.all(np.abs(counts - n * p0) < 4.5 * sd), (counts / n, p0)
    # Acceptance rate at position 0 = sum_v min(p_v, q_v).
    a = np.minimum(p0, q0).sum()
    assert abs(accepted0 - n * a) < 4.5 * np.sqrt(n * a * (1 - a))


def test_stochastic_verify_special_cases():
    rng = np.random.default_rng(12)
    V, P, T = 7, 4, 1.0
    L = rng.normal(size=(3, P, V))
    Z = np.concatenate([L, rng.normal(size=(3, 1, V))], axis=1)  # p_i == q_i for i < P
    draft = rng.integers(0, V, size=(3, P))
    u = rng.uniform(0.01, 0.99, size=(3, P))
    g = -np.log(-np.log(rng.uniform(1e-9, 1 - 1e-9, size=(3, V))))
    acc, adv, nxt, _, _ = O.verify_stochastic(draft, L, Z, u, g, T)
    assert np.all(acc == P) and np.all(adv == P + 1)  # identical distributions: everything accepted
    assert np.array_equal(nxt, np.argmax(Z[:, P] / T + g, -1))  # bonus token ~ p_P by Gumbel-max
    # A draft token the target gives (almost) no mass is rejected, and the
    # residual draw never returns it.
    Z2 = Z.copy()
    Z2[:, 0, :] = 0.0
    Z2[np.arange(3), 0, draft[:, 0]] = -1e4
    acc2, _, nxt2, _, _ = O.verify_stochastic(draft, L, Z2, u, g, T)
    assert np.all(acc2 == 0) and np.all(nxt2 != draft[:, 0])
