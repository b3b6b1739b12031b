"""GPU parity: every entry point, called through the C ABI, against the CPU
oracle on the same seeded inputs. Small cases compare every element; the
full-size workloads compare sampled outputs and whole chains of sampled
requests."""
import numpy as np
import pytest
import torch

import oracle.domino_oracle as O
from draft_head_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from draft_head_gb300 import binding as B
    from tests import parity_log
    from tests.gpu_harness import (GpuCase, TOL, check_logits, compare_forced, compare_tokens, compare_trees,
                                   gpu_candidates, make, oracle_all, small_bf16_cfg, to_dev)


def _tiny(seed, **kw):
    return make(synth.CONFIGS["tiny_f32"], synth.case_seed("tiny_f32", seed), **kw)


# ------------------------------------------------------------------ gate table
@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_gate_table(kind):
    case = _tiny(0) if kind == "f32" else make(small_bf16_cfg(d=328, e=328), 1)
    gc = GpuCase(case)
    ref = O.widen(case["emb"]) @ O.widen(case["w_ih"]).T + O.widen(case["b_ih"])
    got = gc.table.view(case["V"], -1).cpu().numpy()
    tol = 1e-5 if kind == "f32" else 1e-4
    assert np.max(np.abs(got - ref)) < tol


# ------------------------------------------------------------------ base logits
@pytest.mark.parametrize("kind,bs,d", [("f32", 1, 64), ("bf16", 1, 320), ("bf16", 3, 328),
                                       ("bf16", 20, 328)])
def test_base_logits(kind, bs, d):
    case = _tiny(1, batch=bs) if kind == "f32" else make(small_bf16_cfg(d=d, e=d, batch=bs), 2 + bs)
    gc = GpuCase(case)
    L, Ph = gc.base()
    ref = O.base_logits(case["H"], case["w_lm"])
    refp = O.widen(case["H"]) @ O.widen(case["w1"])[:, :case["d"]].T
    tol = 1e-4 if kind == "f32" else 1e-3  # exact bf16 products, fp32 sums
    assert np.max(np.abs(L.cpu().numpy() - ref)) < tol
    assert np.max(np.abs(Ph.cpu().numpy() - refp)) < tol


# ------------------------------------------------------------------ chain, tiny fp32, 20 seeds
@pytest.mark.parametrize("seed", range(20))
def test_chain_tiny_f32(seed):
    case = _tiny(seed)
    gc = GpuCase(case)
    L, Ph = gc.base()
    _, Lo, toks, margins, logits = oracle_all(case)
    gt, _ = gc.chain(L, Ph)
    compare_tokens(gt.cpu().numpy(), toks, margins)
    # forced with the oracle's draft: logits comparable at every position
    gf, glo = gc.chain(L, Ph, force=toks, want_logits=True)
    _, _, tf, mf, lf = oracle_all(case, force=toks)
    check_logits(glo.cpu().numpy(), lf, "f32")
    compare_forced(gf.cpu().numpy(), tf, mf)
    # verify against uniform targets
    tgt = synth.make_targets(toks, "uniform", None, case["V"], seed=case["seed"])
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    adv = torch.empty(1, dtype=torch.int32, device="cuda")
    B.domino_verify(gt, to_dev(tgt), 1, case["P"], acc, adv)
    ra, rv = O.verify(gt.cpu().numpy(), tgt)
    assert acc.item() == ra[0] and adv.item() == rv[0]
    assert gc.status() == 0


# ------------------------------------------------------------------ chain, bf16 small
@pytest.mark.parametrize("bs,temperature,strong,V", [(1, 0.0, False, 1000), (1, 0.0, True, 1000),
                                                     (1, 1.0, False, 1000), (2, 0.0, True, 1000),
                                                     (3, 0.0, True, 1000), (3, 1.0, False, 1000),
                                                     (4, 1.0, True, 1000), (4, 0.0, False, 1000),
                                                     (1, 0.0, True, 1001), (3, 1.0, True, 1003),
                                                     (5, 0.0, True, 1000), (8, 0.0, True, 1000),
                                                     (20, 1.0, True, 1000), (64, 1.0, False, 1000)])
def test_chain_bf16_small(bs, temperature, strong, V):
    # batch <= 4: the small-batch kernel (each batch size is its own
    # instantiation; V % 4 != 0 takes the per-element staging path instead of
    # bulk copies); batch 5-64: the batched tensor-core kernel.
    cfg = small_bf16_cfg(d=328, e=328, batch=bs, temperature=temperature, V=V)
    case = make(cfg, 10 + bs + V, strong_coupling=strong)
    gc = GpuCase(case)
    L, Ph = gc.base()
    _, _, toks, margins, _ = oracle_all(case, temperature=temperature, want_logits=False)
    gt, _ = gc.chain(L, Ph, temperature=temperature)
    compare_tokens(gt.cpu().numpy(), toks, margins)
    gf, glo = gc.chain(L, Ph, temperature=temperature, force=toks, want_logits=True)
    _, _, tf, mf, lf = oracle_all(case, temperature=temperature, force=toks)
    check_logits(glo.cpu().numpy(), lf, "bf16")
    compare_forced(gf.cpu().numpy(), tf, mf)
    assert gc.status() == 0


def test_chain_w2_zero_reproduces_parallel_draft():
    case = make(small_bf16_cfg(d=328, e=328, batch=2), 31, w2_zero=True)
    gc = GpuCase(case)
    L, Ph = gc.base()
    gt, glo = gc.chain(L, Ph, want_logits=True)
    assert torch.equal(glo, L)  # zero correction: L_base exactly
    assert torch.equal(gt.long(), torch.argmax(L, dim=-1))


@pytest.mark.parametrize("bs,V", [(8, 40000), (20, 40000), (40, 100000), (64, 100000)])
def test_batched_chain_ranks_exact_ties_by_first_index(bs, V):
    """W2 = 0 makes every drafted token the argmax of its L_base row (the
    correction vanishes), so rows with many exact copies of their maximum, a
    maximum made of -0.0 and +0.0, rows of -inf and a maximum only in the
    last rows must each give the first index of the maximum ([News] 四: the
    greedy draft; ties go to the lowest id). V = 40000 and 100000 give every
    CTA three and six whole 128-row tiles plus a ragged tail; batch 40 has
    three request chunks of 16; both the plain chain and the draft
    statistics form run the batched kernel at these batches."""
    case = make(small_bf16_cfg(V=V, batch=bs), 71, w2_zero=True)
    gc = GpuCase(case)
    _, Ph = gc.base()
    P, V = gc.P, gc.V
    rng = np.random.default_rng(5)
    L = rng.integers(-6, 3, size=(bs, P, V)).astype(np.float32) * 0.5  # maximum 1.0, ~V / 9 copies
    L[0, 0] = -np.inf
    z = rng.integers(-8, 1, size=V).astype(np.float32)  # maximum 0, of either sign
    z[z == 0] = np.where(rng.random(int((z == 0).sum())) < 0.5, -0.0, 0.0)
    L[0, 1] = z
    L[1 % bs, 2] = -1.0
    L[1 % bs, 2, [V - 3, V - 1]] = 2.0  # only in the last CTA's tail
    L[2 % bs, 3] = -1.0
    L[2 % bs, 3, [4097, 4098, V - 10000]] = 3.0
    L[3 % bs, 4] = 0.25
    L[3 % bs, 4, V // 2] = np.inf  # one +inf
    want = np.argmax(L, axis=-1)
    Ld = to_dev(L)
    toks, _ = gc.chain(Ld, Ph)
    assert np.array_equal(toks.cpu().numpy(), want)
    assert B.domino_draft_chain_stats_supported(gc.head, bs, P)
    st = torch.empty(bs, P, dtype=torch.int32, device="cuda")
    u = torch.empty(bs, P, gc.r, dtype=torch.float32, device="cuda")
    lse = torch.empty(bs, P, dtype=torch.float32, device="cuda")
    B.domino_draft_chain_stats(gc.head, Ld, Ph, gc.anchor, bs, P, 0.0, None, 0, None, st, u, lse, gc.ws)
    assert np.array_equal(st.cpu().numpy(), want)
    assert gc.status() == 0
    # The row log-partitions (T' = 1) where they are finite.
    L64 = L.astype(np.float64)
    m = L64.max(axis=-1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        ref = (m + np.log(np.exp(L64 - m).sum(axis=-1, keepdims=True)))[..., 0]
    fin = np.isfinite(ref)
    assert np.allclose(lse.cpu().numpy()[fin], ref[fin], rtol=0, atol=1e-4)


def test_chain_is_deterministic():
    case = make(small_bf16_cfg(d=328, e=328, batch=1), 33, strong_coupling=True)
    gc = GpuCase(case)
    L, Ph = gc.base()
    a, la = gc.chain(L, Ph, want_logits=True)
    b, lb = gc.chain(L, Ph, want_logits=True)
    assert torch.equal(a, b) and torch.equal(la, lb)


# ------------------------------------------------------------------ verify
def test_verify_edge_cases():
    rng = np.random.default_rng(0)
    for bs, P in [(1, 1), (7, 15), (33, 40), (64, 15)]:
        d = rng.integers(0, 4, size=(bs, P)).astype(np.int32)
        t = d.copy()
        flip = rng.random((bs, P)) < 0.15
        t[flip] += 1
        t[0, :] = d[0, :]          # full accept
        if bs > 1:
            t[1, 0] = d[1, 0] + 1  # reject at once
        acc = torch.empty(bs, dtype=torch.int32, device="cuda")
        adv = torch.empty(bs, dtype=torch.int32, device="cuda")
        B.domino_verify(to_dev(d), to_dev(t), bs, P, acc, adv)
        ra, rv = O.verify(d, t)
        assert np.array_equal(acc.cpu().numpy(), ra) and np.array_equal(adv.cpu().numpy(), rv)
    B.domino_verify(None, None, 0, 15, acc, adv)  # empty batch is a no-op


# ------------------------------------------------------------------ top-M
@pytest.mark.parametrize("rows,n,M", [(3, 1000, 64), (5, 151936, 64), (2, 9000, 256), (4, 70, 70),
                                      (2, 5000, 1)])
def test_topm_select(rows, n, M):
    rng = np.random.default_rng(rows * n)
    vals = rng.integers(-40, 40, size=(rows, n)).astype(np.float32) * 0.125  # many exact ties
    vals[0, 17] = np.float32(-0.0)
    dv = to_dev(vals)
    ids = torch.empty(rows, M, dtype=torch.int32, device="cuda")
    out = torch.empty(rows, M, dtype=torch.float32, device="cuda")
    ws = B.workspace(B.domino_topm_workspace_bytes(rows, n, M))
    B.domino_topm_select(dv, rows, n, M, ids, out, ws)
    for rr in range(rows):
        ref, _ = O.top_m(vals[rr], M)
        assert np.array_equal(ids[rr].cpu().numpy(), ref)
        assert np.array_equal(out[rr].cpu().numpy(), vals[rr][ref])


# ------------------------------------------------------------------ tree
def _tree_gpu(gc, L, Ph, N, M, temperature=0.0):
    bs = gc.bs
    tok = torch.empty(bs, N + 1, dtype=torch.int32, device="cuda")
    par = torch.empty_like(tok)
    dep = torch.empty_like(tok)
    sco = torch.empty(bs, N + 1, dtype=torch.float32, device="cuda")
    B.dominotree_build(gc.head, L, Ph, gc.anchor, bs, gc.P, N, M, tok, par, dep, sco, gc.ws,
                       temperature=temperature)
    return tok.cpu().numpy(), par.cpu().numpy(), dep.cpu().numpy(), sco.cpu().numpy()


def check_tree(g, o, L, N, M, requests):
    """Every listed request under the strict rule of tests/tree_check.py; the
    GPU's own candidate sets decide whether a set difference is real. Returns
    the number of requests compared up to a near tie."""
    exact, ties = compare_trees(g, o, N, requests, gpu_cands=gpu_candidates(L, M))
    parity_log.trees(exact, ties)
    return ties


@pytest.mark.parametrize("kind,bs,N,M,strong,T", [("f32", 1, 16, 8, True, 0.0), ("f32", 2, 10, 64, False, 0.0),
                                                  ("bf16", 3, 16, 64, True, 0.0), ("bf16", 2, 12, 5, True, 0.0),
                                                  ("bf16", 2, 16, 1, False, 0.0), ("bf16", 3, 16, 64, True, 0.5),
                                                  ("f32", 2, 16, 8, True, 0.5), ("bf16", 2, 12, 16, True, 1.0)])
def test_tree(kind, bs, N, M, strong, T):
    if kind == "f32":
        case = _tiny(3, batch=bs, strong_coupling=strong)
    else:
        case = make(small_bf16_cfg(d=328, e=328, batch=bs, block=6 if M == 1 else 16), 40 + M,
                    strong_coupling=strong)
    gc = GpuCase(case, n_nodes=N, top_m=M)
    L, Ph = gc.base()
    g = _tree_gpu(gc, L, Ph, N, M, temperature=T)
    head = O.prepare_head(case)
    Lo = O.base_logits(case["H"], case["w_lm"])
    o = O.tree_build(head, case["H"], Lo, case["anchor"], N, M, temperature=T)
    ties = check_tree(g, o, L, N, M, range(bs))
    assert ties == 0, f"{ties} of {bs} trees differ at an oracle near tie"
    assert gc.status() == 0


# Larger batches and widths: batch 20 (bf16), batch 100 (fewer worker CTAs
# than requests), and g = 1024 in fp32 at batch 40, where the node states do
# not all fit in shared memory at once and are staged in blocks. W_lm is
# scaled by 8 (exact in bf16) so the candidate distributions are peaked and
# the best-first trees go deep (mean depth about 3, up to 10): the states of
# nodes below the root decide the pops.
@pytest.mark.parametrize("kind,bs,N,M", [("bf16", 20, 16, 64), ("f32", 100, 8, 8), ("f32_g1024", 40, 8, 64)])
def test_tree_larger_batches(kind, bs, N, M):
    if kind == "bf16":
        case = make(small_bf16_cfg(d=328, e=328, batch=bs), 70 + bs, strong_coupling=True)
        case["w_lm"] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(case["w_lm"]) * 8.0)
    else:
        cfg = dict(synth.CONFIGS["tiny_f32"], block=8)
        if kind == "f32_g1024":
            cfg.update(g=1024, r=256, block=16)
        case = make(cfg, synth.case_seed("tiny_f32", bs), batch=bs, strong_coupling=True)
        case["w_lm"] = (case["w_lm"] * 8.0).astype(np.float32)
    gc = GpuCase(case, n_nodes=N, top_m=M)
    L, Ph = gc.base()
    g = _tree_gpu(gc, L, Ph, N, M)
    head = O.prepare_head(case)
    Lo = O.base_logits(case["H"], case["w_lm"])
    o = O.tree_build(head, case["H"], Lo, case["anchor"], N, M)
    ties = check_tree(g, o, L, N, M, range(bs))
    assert ties == 0, f"{ties} of {bs} trees differ at an oracle near tie"
    assert gc.status() == 0


# ------------------------------------------------------------------ bounded waits
def test_wait_timeout_is_reported_not_hung():
    ws = B.workspace(4096)
    ws.zero_()
    B.domino_selftest_wait_timeout(2_000_000, ws)  # 2 ms bound on a flag nothing sets
    assert B.domino_last_status(ws) == 4            # DOMINO_ERR_TIMEOUT
    assert B.domino_last_status(ws) == 0            # cleared by the read
    # The context stays usable afterwards.
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


# ------------------------------------------------------------------ fixed-point range
# The bottleneck sums W1_s S cross CTAs as 64-bit fixed-point integers. A W1_s
# whose partial sums could carry an accumulator past its range must come back
# as a device data error, never as tokens with DOMINO_OK.
@pytest.mark.parametrize("kind", ["bf16_small", "f32_generic", "bf16_tree"])
def test_fixed_point_range_is_reported(kind):
    if kind == "f32_generic":
        case = _tiny(5)
        scale = 1e9
    else:
        case = make(small_bf16_cfg(d=320, e=320, batch=2), 77, strong_coupling=True)
        scale = 3e4
    d = case["d"]
    w1 = synth.as_f32(case["w1"]).copy()
    w1[:, d:] = np.sign(w1[:, d:] + 1e-30) * scale  # |W1_s| = scale everywhere
    case["w1"] = w1.astype(np.float32) if case["w1"].dtype != np.uint16 else synth.f32_to_bf16_bits(w1)
    N, M = (8, 16) if kind == "bf16_tree" else (0, 0)
    gc = GpuCase(case, n_nodes=N, top_m=M)
    L, Ph = gc.base()
    assert gc.status() == 0
    if kind == "bf16_tree":
        _tree_gpu(gc, L, Ph, N, M)
    else:
        gc.chain(L, Ph)
    assert gc.status() == 6  # DOMINO_ERR_DEVICE_DATA
    # The same case with the original scale of W1_s runs clean afterwards.
