"""GPU parity for tree acceptance and the head-off baselines, through the C ABI,
against the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle.domino_oracle as O
from draft_head_gb300 import binding as B
from draft_head_gb300 import synth
from tests import parity_log
from tests.gpu_harness import (NEAR_TIE, GpuCase, _draw_within_fp32_error, compare_trees, gpu_candidates, make,
                               small_bf16_cfg, to_dev)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ tree acceptance
def random_trees(bs, N, V, seed, fill=None):
    """Valid trees: parents precede children, sibling tokens distinct, slots
    past `fill` empty (a tree that ran dry)."""
    rng = np.random.default_rng(seed)
    tok = np.full((bs, N + 1), -1, np.int32)
    par = np.full((bs, N + 1), -1, np.int32)
    for b in range(bs):
        n = N if fill is None else fill
        tok[b, 0] = rng.integers(0, V)
        kids = {}
        for k in range(1, n + 1):
            open_parents = [q for q in range(k) if len(kids.get(q, ())) < V]
            p = open_parents[int(rng.integers(0, len(open_parents)))]
            used = kids.setdefault(p, set())
            free = [t for t in range(V) if t not in used]
            t = free[int(rng.integers(0, len(free)))]
            used.add(t)
            tok[b, k], par[b, k] = t, p
    return tok, par


def tree_verify_gpu(tok, par, tgt, want_mask=True):
    bs, n1 = tok.shape
    acc = torch.empty(bs, dtype=torch.int32, device="cuda")
    adv = torch.empty_like(acc)
    path = torch.empty(bs, n1, dtype=torch.int32, device="cuda")
    mask = torch.empty(bs, n1, n1, dtype=torch.uint8, device="cuda") if want_mask else None
    B.dominotree_verify(to_dev(tok), to_dev(par), to_dev(tgt), bs, n1 - 1, acc, adv, path, mask)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), adv.cpu().numpy(), path.cpu().numpy(), (mask.cpu().numpy() if want_mask else None)


@pytest.mark.parametrize("bs,N,V,fill,p", [(200, 16, 4, None, 0.3), (37, 64, 9, None, 0.1), (50, 1, 3, None, 0.5),
                                          (64, 40, 5, 17, 0.2), (5, 64, 2, None, 0.0)])
def test_tree_verify_random_trees(bs, N, V, fill, p):
    tok, par = random_trees(bs, N, V, seed=bs * 7 + N, fill=fill)
    tgt = synth.make_tree_targets(tok, par, p, V, seed=N)
    acc, adv, path, mask = tree_verify_gpu(tok, par, tgt)
    oa, oad, op, om = O.tree_verify(tok, par, tgt)
    assert np.array_equal(acc, oa) and np.array_equal(adv, oad)
    assert np.array_equal(path, op)
    assert np.array_equal(mask, om)
    if p == 0.0:
        assert np.all(acc >= 1)  # the target always follows the first-popped child


def test_tree_verify_on_oracle_trees_and_no_mask():
    case = make(small_bf16_cfg(d=320, e=320, batch=3), 61, strong_coupling=True)
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"])
    tr = O.tree_build(head, case["H"], L, case["anchor"], 16, 8)
    tok, par = tr["node_token"].astype(np.int32), tr["node_parent"].astype(np.int32)
    tgt = synth.make_tree_targets(tok, par, 0.2, case["V"], seed=61)
    acc, adv, path, _ = tree_verify_gpu(tok, par, tgt, want_mask=False)
    oa, oad, op, _ = O.tree_verify(tok, par, tgt)
    assert np.array_equal(acc, oa) and np.array_equal(adv, oad) and np.array_equal(path, op)


def test_tree_verify_empty_batch_and_bad_args():
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dominotree_verify(z, z, z, 0, 4, z, z)  # batch 0: nothing to do
    with pytest.raises(B.DominoError):
        B.dominotree_verify(None, z, z, 1, 4, z, z)


# ------------------------------------------------------------------ head-off chain
def headoff_gpu(L, T, g, gstride, ws=None):
    bs, P, V = L.shape
    Ld = to_dev(L)
    toks = torch.empty(bs, P, dtype=torch.int32, device="cuda")
    if ws is None:
        ws = B.workspace(B.domino_headoff_workspace_bytes(bs, P, V))
    B.domino_draft_chain_headoff(Ld, bs, P, V, T, g, gstride, toks, ws)
    torch.cuda.synchronize()
    assert B.domino_last_status(ws) == 0
    return toks.cpu().numpy(), ws


@pytest.mark.parametrize("bs,P,V,T", [(1, 15, 1000, 0.0), (3, 7, 8192, 0.0), (4, 5, 20000, 1.0),
                                     (2, 3, 17, 0.5), (64, 15, 4099, 1.0)])
def test_headoff_chain(bs, P, V, T):
    L = synth.normal((bs, P, V), 1.0, 7000 + V, 0)
    g_full = synth.gumbel_noise((bs, P + 1, V), 7000 + V) if T > 0 else None
    gd = to_dev(g_full)[:, 1:, :] if T > 0 else None
    gstride = (P + 1) * V if T > 0 else 0
    toks, ws = headoff_gpu(L, T, gd, gstride)
    ot, om = O.draft_chain_headoff(L.astype(np.float64), T, g_full[:, 1:, :] if T > 0 else None)
    bad = (toks != ot) & ~(om < NEAR_TIE)
    assert not bad.any(), np.argwhere(bad)[:5]
    if T == 0.0:
        assert np.array_equal(toks, ot)  # decisions on exact fp32 values
    # The workspace is left clean: a second call gives the same tokens.
    toks2, _ = headoff_gpu(L, T, gd, gstride, ws)
    assert np.array_equal(toks, toks2)


def test_headoff_chain_equals_w2_zero_chain_on_gpu():
    case = make(small_bf16_cfg(batch=2), 62, w2_zero=True)
    gc = GpuCase(case)
    L, Ph = gc.base()
    full = gc.chain(L, Ph)[0].cpu().numpy()
    bs, P, V = case["batch"], case["P"], case["V"]
    toks = torch.empty(bs, P, dtype=torch.int32, device="cuda")
    ws = B.workspace(B.domino_headoff_workspace_bytes(bs, P, V))
    B.domino_draft_chain_headoff(L, bs, P, V, 0.0, None, 0, toks, ws)
    assert np.array_equal(toks.cpu().numpy(), full)


# ------------------------------------------------------------------ marginal tree
def marginal_gpu(L, anchor, N, M, temperature=0.0):
    bs, P, V = L.shape
    shape = (bs, N + 1)
    out = [torch.empty(shape, dtype=torch.int32, device="cuda") for _ in range(3)]
    sc = torch.empty(shape, dtype=torch.float32, device="cuda")
    ws = B.workspace(B.domino_headoff_workspace_bytes(bs, P, V, N, M))
    B.dominotree_build_marginal(to_dev(L), to_dev(anchor), bs, P, V, N, M, out[0], out[1], out[2], sc, ws,
                                temperature=temperature)
    torch.cuda.synchronize()
    assert B.domino_last_status(ws) == 0
    return tuple(x.cpu().numpy() for x in out) + (sc.cpu().numpy(),)


@pytest.mark.parametrize("bs,P,V,N,M,T", [(4, 15, 1000, 16, 64, 0.0), (2, 6, 500, 64, 5, 0.0),
                                         (3, 15, 3000, 16, 256, 0.0), (2, 4, 50, 16, 1, 0.0),
                                         (1, 2, 7, 64, 3, 0.0), (4, 15, 1000, 16, 64, 0.5),
                                         (2, 6, 500, 64, 5, 1.0)])
def test_marginal_tree(bs, P, V, N, M, T):
    L = synth.normal((bs, P, V), 1.0, 8000 + V, 0)
    anchor = np.arange(bs, dtype=np.int32) % V
    g = marginal_gpu(L, anchor, N, M, temperature=T)
    o = O.tree_build_marginal(L.astype(np.float64), anchor, N, M, temperature=T)
    exact, ties = compare_trees(g, o, N, range(bs), gpu_cands=gpu_candidates(to_dev(L), M))
    parity_log.trees(exact, ties)
    assert ties == 0


def test_marginal_tree_equals_conditional_tree_with_w2_zero():
    case = make(small_bf16_cfg(d=320, e=320, batch=2), 63, w2_zero=True)
    N, M = 16, 16
    gc = GpuCase(case, n_nodes=N, top_m=M)
    L, Ph = gc.base()
    bs, P, V = case["batch"], case["P"], case["V"]
    shape = (bs, N + 1)
    cond = [torch.empty(shape, dtype=torch.int32, device="cuda") for _ in range(3)]
    csc = torch.empty(shape, dtype=torch.float32, device="cuda")
    B.dominotree_build(gc.head, L, Ph, gc.anchor, bs, P, N, M, cond[0], cond[1], cond[2], csc, gc.ws)
    anchor = case["anchor"].astype(np.int32)
    g = marginal_gpu(L.cpu().numpy().astype(np.float32), anchor, N, M)
    for k in range(3):
        assert np.array_equal(g[k], cond[k].cpu().numpy())
    assert np.array_equal(g[3], csc.cpu().numpy())


# ------------------------------------------------------------------ whole-cycle graph
def test_graph_captured_cycle_matches_eager():
    """The base pass, the chain and verify captured as one CUDA graph give the
    eager results, and a replay reads new inputs copied into the same buffers."""
    from draft_head_gb300.runtime import DominoDrafter
    case = make(small_bf16_cfg(batch=1), 64, strong_coupling=True)
    w = {k: to_dev(case[k]) for k in ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2")}
    P = case["P"]
    dr = DominoDrafter(w, 1, P)
    H = to_dev(case["H"])
    anchor = to_dev(case["anchor"].astype(np.int32))
    target = to_dev(synth.make_targets(np.zeros((1, P), np.int64), "uniform", None, case["V"], seed=2))
    dr.draft(H, anchor)
    dr.verify(target)
    eager_t, eager_a = dr.tokens.clone(), dr.accept.clone()
    dr.capture_cycle(H, anchor, target)
    dr.tokens.fill_(-7)
    dr.replay()
    torch.cuda.synchronize()
    assert torch.equal(dr.tokens, eager_t) and torch.equal(dr.accept, eager_a)
    # New inputs in the captured buffers.
    case2 = make(small_bf16_cfg(batch=1), 65, strong_coupling=True)
    H.copy_(to_dev(case2["H"]))
    anchor.copy_(to_dev(case2["anchor"].astype(np.int32)))
    dr.replay()
    torch.cuda.synchronize()
    got = dr.tokens.clone()
    dr.draft(H, anchor)
    torch.cuda.synchronize()
    assert torch.equal(got, dr.tokens)
    assert dr.last_status() == 0


def _capture(step):
    """step() run once on a side stream, then captured as one CUDA graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


def test_graph_captured_tree_and_sampled_steps_match_eager():
    """The benchmark's other steps captured as one graph each give the eager
    results: base pass + DominoTree build + tree acceptance (cooperative tree
    kernel, three top-M passes), and base pass + Gumbel chain with its logits +
    verification at T = 1 (one thread-block cluster per request)."""
    from draft_head_gb300.runtime import DominoDrafter
    # Tree: batch 3, N = 8, M = 16.
    case = make(small_bf16_cfg(batch=3), 66, strong_coupling=True)
    w = {k: to_dev(case[k]) for k in ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2")}
    P, V = case["P"], case["V"]
    dr = DominoDrafter(w, 3, P, 8, 16)
    H = to_dev(case["H"])
    anchor = to_dev(case["anchor"].astype(np.int32))
    tnext = to_dev(synth.make_targets(np.zeros((3, 9), np.int64), "uniform", None, V, seed=6))

    def tree_step():
        dr.base(H)
        dr.tree(anchor)
        dr.tree_verify(tnext, want_path=True, want_mask=True)

    tree_step()
    torch.cuda.synchronize()
    eager = [x.clone() for x in (dr.node_token, dr.node_parent, dr.node_depth, dr.node_score, dr.accept,
                                 dr.tree_path, dr.tree_mask)]
    g = _capture(tree_step)
    for x in (dr.node_token, dr.node_parent, dr.accept):
        x.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    got = (dr.node_token, dr.node_parent, dr.node_depth, dr.node_score, dr.accept, dr.tree_path, dr.tree_mask)
    for a, b in zip(got, eager):
        assert torch.equal(a, b)
    assert dr.last_status() == 0

    # Gumbel chain with logits out and verification at T = 1, batch 8.
    bs = 8
    case = make(small_bf16_cfg(batch=bs, temperature=1.0), 67, strong_coupling=True)
    w = {k: to_dev(case[k]) for k in ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2")}
    dr = DominoDrafter(w, bs, P)
    H = to_dev(case["H"])
    anchor = to_dev(case["anchor"].astype(np.int32))
    gm = to_dev(case["gumbel"])
    Z = to_dev((synth.normal((bs, P + 1, V), 1.0, 68, 0)).astype(np.float32))
    U = to_dev(synth.uniform_open01((bs, P), 68, 1).astype(np.float32))
    G = to_dev(synth.gumbel_noise((bs, V), 69))

    def sampled_step():
        dr.base(H)
        dr.chain(anchor, 1.0, gm[:, 1:, :], (P + 1) * V, logits_out=dr.draft_logits())
        dr.verify_sampled(Z, U, G, 1.0)

    sampled_step()
    torch.cuda.synchronize()
    eager = [x.clone() for x in (dr.tokens, dr.draft_logits(), dr.accept, dr.advanced, dr.next_token)]
    g = _capture(sampled_step)
    for x in (dr.tokens, dr.accept, dr.next_token):
        x.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    got = (dr.tokens, dr.draft_logits(), dr.accept, dr.advanced, dr.next_token)
    for a, b in zip(got, eager):
        assert torch.equal(a, b)
    assert dr.last_status() == 0


def test_packed_host_io_cycle_matches_eager():
    """The cycle through packed pinned buffers (one copy each way), eager and
    captured as one graph, gives the eager device results."""
    from draft_head_gb300.runtime import DominoDrafter, HostIO
    case = make(small_bf16_cfg(batch=2), 70, strong_coupling=True)
    w = {k: to_dev(case[k]) for k in ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2")}
    P, V, d = case["P"], case["V"], case["d"]
    dr = DominoDrafter(w, 2, P)
    H = to_dev(case["H"])
    anchor = to_dev(case["anchor"].astype(np.int32))
    tgt = synth.make_targets(np.zeros((2, P), np.int64), "uniform", None, V, seed=3)
    dr.draft(H, anchor)
    dr.verify(to_dev(tgt))
    torch.cuda.synchronize()
    eager_t, eager_a = dr.tokens.cpu(), dr.accept.cpu()
    io = HostIO(dr, d, H.dtype)
    io.H_host.copy_(H.cpu())
    io.anchor_host.copy_(anchor.cpu())
    io.target_host.copy_(torch.from_numpy(tgt))
    dr.cycle_io(io)
    torch.cuda.synchronize()
    assert torch.equal(io.tokens_host, eager_t) and torch.equal(io.accept_host, eager_a)
    io.host_out.fill_(-7)
    dr.capture_io_cycle(io)
    io.host_out.fill_(-7)
    dr.replay_io_cycle()
    torch.cuda.synchronize()
    assert torch.equal(io.tokens_host, eager_t) and torch.equal(io.accept_host, eager_a)
    assert dr.last_status() == 0


def test_graph_captured_host_cycle_matches_eager():
    """The whole host cycle (pinned inputs copied in, base pass, chain, verify,
    results copied out) captured as one graph gives the eager results, and a
    replay picks up new contents of the pinned input buffers."""
    from draft_head_gb300.runtime import DominoDrafter
    case = make(small_bf16_cfg(batch=1), 66, strong_coupling=True)
    w = {k: to_dev(case[k]) for k in ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2")}
    P, V = case["P"], case["V"]
    dr = DominoDrafter(w, 1, P)
    pinned = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    Hh = pinned(case["H"].view(np.int16)).view(torch.bfloat16)
    ah = pinned(case["anchor"].astype(np.int32))
    th = pinned(synth.make_targets(np.zeros((1, P), np.int64), "uniform", None, V, seed=3))
    tok_h = torch.empty(1, P, dtype=torch.int32).pin_memory()
    acc_h = torch.empty(1, dtype=torch.int32).pin_memory()
    Hd = torch.empty(Hh.shape, dtype=torch.bfloat16, device="cuda")
    ad = torch.empty(1, dtype=torch.int32, device="cuda")
    td = torch.empty(1, P, dtype=torch.int32, device="cuda")
    dr.cycle_from_host(Hh, ah, th, tok_h, acc_h, Hd, ad, td)
    torch.cuda.synchronize()
    eager_t, eager_a = tok_h.clone(), acc_h.clone()
    dr.capture_host_cycle(Hh, ah, th, tok_h, acc_h, Hd, ad, td)
    tok_h.fill_(-7)
    dr.replay_host_cycle()
    torch.cuda.synchronize()
    assert torch.equal(tok_h, eager_t) and torch.equal(acc_h, eager_a)
    case2 = make(small_bf16_cfg(batch=1), 67, strong_coupling=True)
    Hh.copy_(torch.from_numpy(case2["H"].view(np.int16)).view(torch.bfloat16))
    ah.copy_(torch.from_numpy(case2["anchor"].astype(np.int32)))
    dr.replay_host_cycle()
    torch.cuda.synchronize()
    got_t, got_a = tok_h.clone(), acc_h.clone()
    dr.cycle_from_host(Hh, ah, th, tok_h, acc_h, Hd, ad, td)
    torch.cuda.synchronize()
    assert torch.equal(got_t, tok_h) and torch.equal(got_a, acc_h)
    assert dr.last_status() == 0


# ------------------------------------------------------------------ verification at T > 0
def _sampled_inputs(bs, P, V, T, seed, spread=0.5):
    L = synth.normal((bs, P, V), 1.0, seed, 0)
    Z = np.concatenate([L, synth.normal((bs, 1, V), 1.0, seed, 1)], axis=1) + synth.normal((bs, P + 1, V), spread,
                                                                                              seed, 2)
    Z = Z.astype(np.float32)
    g_draft = synth.gumbel_noise((bs, P, V), seed + 1)
    draft = np.argmax(L / T + g_draft, -1).astype(np.int32)  # drafts drawn from q
    U = synth.uniform_open01((bs, P), seed, 3).astype(np.float32)
    G = synth.gumbel_noise((bs, V), seed + 2)
    return draft, L, Z, U, G


def sampled_gpu(draft, L, Z, U, G, T):
    bs, P, V = L.shape
    acc = torch.empty(bs, dtype=torch.int32, device="cuda")
    adv = torch.empty_like(acc)
    nxt = torch.empty_like(acc)
    ws = B.workspace(B.domino_verify_sampled_workspace_bytes(bs, P))
    B.domino_verify_sampled(to_dev(draft), to_dev(L), to_dev(Z), to_dev(U), to_dev(G), bs, P, V, T, acc, adv, nxt,
                            ws)
    torch.cuda.synchronize()
    assert B.domino_last_status(ws) == 0
    return acc.cpu().numpy(), adv.cpu().numpy(), nxt.cpu().numpy()


# The cases cover clusters of 1, 2, 4 and 8 CTAs per request (the library picks
# K from the batch and V), the scalar path with K > 1 (V % 4 != 0), and walks
# that run deep or to the end (target logits close to the draft's).
@pytest.mark.parametrize("bs,P,V,T,spread", [(16, 7, 1000, 1.0, 0.5), (8, 15, 4099, 0.5, 0.3), (32, 3, 17, 1.0, 2.0),
                                            (4, 15, 151936, 1.0, 0.5), (160, 3, 16384, 1.0, 0.5),
                                            (100, 2, 32768, 0.7, 0.5), (2, 6, 16387, 1.0, 0.4),
                                            (8, 15, 32768, 1.0, 0.05), (3, 0, 1000, 1.0, 0.5), (5, 4, 1, 1.0, 0.5),
                                            (64, 15, 151936, 1.0, 0.5)])
def test_verify_sampled(bs, P, V, T, spread):
    draft, L, Z, U, G = _sampled_inputs(bs, P, V, T, 9300 + V, spread)
    acc, adv, nxt = sampled_gpu(draft, L, Z, U, G, T)
    oa, oad, on, rm, tm = O.verify_stochastic(draft, L, Z, U, G, T)
    ties = bounded = 0
    for b in range(bs):
        if acc[b] != oa[b]:
            # The acceptance test U < p(x) / q(x): the fp32 ratio is within 1e-5
            # of the exact one, so only a draw this close to it can flip.
            assert rm[b] < 1e-4, f"b={b}: accept {acc[b]} vs {oa[b]}, margin {rm[b]}"
            ties += 1
            continue
        assert adv[b] == oad[b]
        if nxt[b] != on[b]:
            if tm[b] < NEAR_TIE:
                ties += 1
            else:
                assert _draw_within_fp32_error(L[b], Z[b], G[b], int(oa[b]), int(on[b]), int(nxt[b]), T), (
                    f"b={b}: token {nxt[b]} vs {on[b]}, margin {tm[b]}")
                bounded += 1
    parity_log.tokens(bs - ties - bounded, ties)
    parity_log.count("sampled_draws_within_fp32_bound", bounded)


def test_verify_sampled_empty_batch():
    """batch 0 is a no-op that succeeds."""
    ws = B.workspace(B.domino_verify_sampled_workspace_bytes(0, 4))
    one = torch.zeros(1, dtype=torch.int32, device="cuda")
    f = torch.zeros(4, dtype=torch.float32, device="cuda")
    B.domino_verify_sampled(one, f, f, f, f, 0, 4, 1, 1.0, one, one, one, ws)
    torch.cuda.synchronize()
    assert B.domino_last_status(ws) == 0


def test_verify_sampled_is_lossless_on_gpu():
    """20000 independent requests of one call: the first emitted token follows
    the target's p_0 (the property the pages claim), and the acceptance rate at
    position 0 is sum_v min(p_v, q_v)."""
    bs, P, V, T = 20000, 2, 5, 0.8
    rng = np.random.default_rng(21)
    l0 = rng.normal(size=(P, V)).astype(np.float32)
    z0 = rng.normal(size=(P + 1, V)).astype(np.float32)
    L = np.broadcast_to(l0, (bs, P, V)).copy()
    Z = np.broadcast_to(z0, (bs, P + 1, V)).copy()
    q0 = np.exp(l0[0].astype(np.float64) / T); q0 /= q0.sum()
    p0 = np.exp(z0[0].astype(np.float64) / T); p0 /= p0.sum()
    g_draft = synth.gumbel_noise((bs, P, V), 77)
    draft = np.argmax(L / T + g_draft, -1).astype(np.int32)
    U = synth.uniform_open01((bs, P), 77, 3).astype(np.float32)
    G = synth.gumbel_noise((bs, V), 78)
    acc, _, nxt = sampled_gpu(draft, L, Z, U, G, T)
    first = np.where(acc >= 1, draft[:, 0], nxt)
    counts = np.bincount(first, minlength=V)
    sd = np.sqrt(bs * p0 * (1 - p0))
    assert np.all(np.abs(counts - bs * p0) < 4.5 * sd), (counts / bs, p0)
    a = np.minimum(p0, q0).sum()
    assert abs((acc >= 1).sum() - bs * a) < 4.5 * np.sqrt(bs * a * (1 - a))
