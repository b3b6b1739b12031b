"""GPU parity of the logits-free sampled path, through the C ABI: the batched
chain's draft statistics (u_i and the row log-partitions of L_i / T) and the
sampled verification that works from them (the head form), against the
oracle (draft_chain_stats, verify_stochastic) on the same seeded inputs, and
against the logits form of the same verification."""
import numpy as np
import pytest
import torch

import oracle.domino_oracle as O
from draft_head_gb300 import binding as B
from draft_head_gb300 import synth
from tests import parity_log
from tests.gpu_harness import (NEAR_TIE, GpuCase, _draw_within_fp32_error, check_logits, compare_forced, make,
                               small_bf16_cfg, to_dev)

pytestmark = pytest.mark.gpu

# u_i is SiLU of a bf16-operand product with fp32 accumulation (S in a high and
# a low bf16 part): well inside 1e-4 at these magnitudes. The log-partition
# sums V terms in fp32 over fp32 logits within the bf16 logit bar.
U_TOL = 1e-4
LSE_TOL = 1e-4


def stats_gpu(gc, L, Ph, T, force=None):
    bs, P = gc.bs, gc.P
    toks = torch.empty(bs, P, dtype=torch.int32, device="cuda")
    u = torch.empty(bs, P, gc.r, dtype=torch.float32, device="cuda")
    lse = torch.empty(bs, P, dtype=torch.float32, device="cuda")
    g, stride = (gc.gumbel[:, 1:, :], gc.gumbel.shape[1] * gc.V) if T > 0 else (None, 0)
    f = to_dev(np.asarray(force, dtype=np.int32)) if force is not None else None
    B.domino_draft_chain_stats(gc.head, L, Ph, gc.anchor, bs, P, T, g, stride, f, toks, u, lse, gc.ws)
    return toks, u, lse


def oracle_forced(case, gpu_toks, T):
    """The oracle chain teacher-forced with the GPU's drafted tokens (the same
    GRU path even where a near tie sent the GPU another way): tokens, margins,
    logits, u, lse."""
    head = O.prepare_head(case)
    Lb = O.base_logits(case["H"], case["w_lm"])
    G = case["gumbel"][:, 1:, :] if T > 0 else None
    toks, margins, logits = O.draft_chain(head, case["H"], Lb, case["anchor"], temperature=T, gumbel=G,
                                          force=gpu_toks, want_logits=True)
    st, _, us, lse = O.draft_chain_stats(head, case["H"], Lb, case["anchor"], temperature=T, gumbel=G,
                                         force=gpu_toks)
    assert np.array_equal(st, toks)
    return toks, margins, logits, us, lse


# Batches 5..64 (the tensor-core chain), greedy and sampled, V = 1000 (one
# ragged tile per CTA) and V = 40000 (three tiles per CTA, the last ragged).
# Batch 40: three request chunks of 16 (six staging slots).
@pytest.mark.parametrize("bs,T,V", [(5, 1.0, 1000), (20, 0.7, 1000), (64, 1.0, 1000), (8, 0.0, 1000),
                                    (12, 1.3, 40000), (40, 1.0, 40000), (1, 1.0, 1000), (3, 0.6, 40000)])
def test_chain_stats(bs, T, V):
    case = make(small_bf16_cfg(batch=bs, V=V, temperature=T), 400 + bs, strong_coupling=True)
    gc = GpuCase(case)
    assert B.domino_draft_chain_stats_supported(gc.head, bs, gc.P)
    L, Ph = gc.base()
    toks, u, lse = stats_gpu(gc, L, Ph, T)
    # The same chain without statistics: the same tokens, bit for bit (at
    # batch <= 4 that call runs the small-batch kernel: equal up to near ties).
    gt = toks.cpu().numpy()
    toks2, logits = gc.chain(L, Ph, T, force=gt, want_logits=True)  # the statistics' GRU path
    torch.cuda.synchronize()
    assert gc.status() == 0
    if bs >= 5:
        assert torch.equal(toks, toks2)
    ot, om, ol, ou, olse = oracle_forced(case, gt, T)
    compare_forced(gt, ot, om)
    check_logits(logits.cpu().numpy(), ol, "bf16")
    du = float(np.max(np.abs(u.cpu().numpy().astype(np.float64) - ou)))
    dl = float(np.max(np.abs(lse.cpu().numpy().astype(np.float64) - olse)))
    parity_log.logits("u", du)
    parity_log.logits("lse", dl)
    assert du < U_TOL, du
    assert dl < LSE_TOL, dl
    # The log-partition of the logits of the plain chain on the same path
    # (fp64 on the host; at batch <= 4 another kernel computed them).
    tau = T if T > 0 else 1.0
    lg = logits.cpu().numpy().astype(np.float64) / tau
    m = lg.max(-1, keepdims=True)
    own = (m + np.log(np.exp(lg - m).sum(-1, keepdims=True)))[..., 0]
    assert float(np.max(np.abs(lse.cpu().numpy() - own))) < (2e-5 if bs >= 5 else 5e-5)


def test_chain_stats_teacher_forced():
    """Forced GRU inputs: the statistics follow the forced path (the oracle
    chain forced with the same tokens)."""
    bs, T = 10, 0.8
    case = make(small_bf16_cfg(batch=bs, temperature=T), 431, strong_coupling=True)
    gc = GpuCase(case)
    L, Ph = gc.base()
    force = synth.normal((bs, gc.P), 1.0, 432, 0)
    force = (np.abs(force) * 1000).astype(np.int64) % gc.V
    toks, u, lse = stats_gpu(gc, L, Ph, T, force=force)
    torch.cuda.synchronize()
    assert gc.status() == 0
    ot, om, ol, ou, olse = oracle_forced(case, force, T)
    compare_forced(toks.cpu().numpy(), ot, om)
    assert float(np.max(np.abs(u.cpu().numpy() - ou))) < U_TOL
    assert float(np.max(np.abs(lse.cpu().numpy() - olse))) < LSE_TOL


def test_chain_stats_unsupported_shapes():
    """Only the tensor-core chain keeps statistics: an fp32 head, or a
    vocabulary that is not a multiple of 4, is refused."""
    case = make(small_bf16_cfg(batch=3, temperature=1.0, V=1002), 31)
    gc = GpuCase(case)
    assert not B.domino_draft_chain_stats_supported(gc.head, 3, gc.P)
    L, Ph = gc.base()
    with pytest.raises(B.DominoError) as e:
        stats_gpu(gc, L, Ph, 1.0)
    assert e.value.status == 2
    from tests.gpu_harness import small_bf16_cfg as _cfg
    f32 = make(dict(_cfg(batch=8, temperature=1.0), dtype="f32"), 32)
    assert not B.domino_draft_chain_stats_supported(GpuCase(f32).head, 8, f32["P"])


def head_verify_gpu(gc, toks, L, u, lse, Z, U, G, T, ws=None):
    bs, P = gc.bs, gc.P
    acc = torch.empty(bs, dtype=torch.int32, device="cuda")
    adv = torch.empty_like(acc)
    nxt = torch.empty_like(acc)
    if ws is None:
        ws = B.workspace(B.domino_verify_sampled_head_workspace_bytes(bs, P))
    B.domino_verify_sampled_head(gc.head, toks, L, u, lse, Z, U, G, bs, P, T, acc, adv, nxt, ws)
    torch.cuda.synchronize()
    assert B.domino_last_status(ws) == 0
    return acc.cpu().numpy(), adv.cpu().numpy(), nxt.cpu().numpy()


def logits_verify_gpu(toks, logits, Z, U, G, T):
    bs, P, V = logits.shape
    acc = torch.empty(bs, dtype=torch.int32, device="cuda")
    adv = torch.empty_like(acc)
    nxt = torch.empty_like(acc)
    ws = B.workspace(B.domino_verify_sampled_workspace_bytes(bs, P))
    B.domino_verify_sampled(toks, logits, Z, U, G, bs, P, V, T, acc, adv, nxt, ws)
    torch.cuda.synchronize()
    assert B.domino_last_status(ws) == 0
    return acc.cpu().numpy(), adv.cpu().numpy(), nxt.cpu().numpy()


def check_against_oracle(acc, adv, nxt, toks, ol, Z, U, G, T, eps_q):
    """The sampled-verification bar: accept lengths equal unless the draw U
    sits within 1e-4 of the oracle's ratio; drawn tokens equal unless the
    oracle's draw margin is a near tie or the GPU's token scores within the
    fp32 error bound. Returns (exact, ties, bounded)."""
    oa, oad, on, rm, tm = O.verify_stochastic(toks, ol, Z, U, G, T)
    ties = bounded = 0
    for b in range(len(acc)):
        if acc[b] != oa[b]:
            assert rm[b] < 1e-4, f"b={b}: accept {acc[b]} vs {oa[b]}, margin {rm[b]}"
            ties += 1
            continue
        assert adv[b] == oad[b]
        if nxt[b] != on[b]:
            if tm[b] < NEAR_TIE:
                ties += 1
            else:
                assert _draw_within_fp32_error(ol[b], Z[b], G[b], int(oa[b]), int(on[b]), int(nxt[b]), T,
                                               eps_q=eps_q), f"b={b}: token {nxt[b]} vs {on[b]}, margin {tm[b]}"
                bounded += 1
    return len(acc) - ties - bounded, ties, bounded


# Spread 0.05: the target follows the draft closely (long accepted runs, some
# requests accept all P); spread 1.5: early rejections, residual draws.
@pytest.mark.parametrize("bs,T,V,spread", [(5, 1.0, 1000, 0.05), (20, 0.7, 1000, 1.5), (64, 1.0, 1000, 0.3),
                                           (64, 1.0, 1000, 0.05), (12, 1.3, 40000, 1.0), (9, 0.5, 40000, 0.05),
                                           (1, 1.0, 1000, 1.0), (2, 0.8, 40000, 0.05)])
def test_verify_sampled_head(bs, T, V, spread):
    case = make(small_bf16_cfg(batch=bs, V=V, temperature=T), 500 + bs, strong_coupling=True)
    gc = GpuCase(case)
    P = gc.P
    L, Ph = gc.base()
    toks, u, lse = stats_gpu(gc, L, Ph, T)
    gt = toks.cpu().numpy()
    _, logits = gc.chain(L, Ph, T, force=gt, want_logits=True)  # the statistics' GRU path
    torch.cuda.synchronize()
    assert gc.status() == 0
    ot, om, ol, _, _ = oracle_forced(case, gt, T)
    dL = check_logits(logits.cpu().numpy(), ol, "bf16")
    seed = 600 + bs
    Zn = np.concatenate([ol.astype(np.float32), synth.normal((bs, 1, V), 1.0, seed, 1)], axis=1)
    Z = (Zn + synth.normal((bs, P + 1, V), spread, seed, 2)).astype(np.float32)
    U = synth.uniform_open01((bs, P), seed, 3).astype(np.float32)
    G = synth.gumbel_noise((bs, V), seed + 2)
    Zd, Ud, Gd = to_dev(Z), to_dev(U), to_dev(G)
    acc, adv, nxt = head_verify_gpu(gc, toks, L, u, lse, Zd, Ud, Gd, T)
    # q's relative error: the kernel's own logit error over T, plus fp32.
    eps_q = 2.0 * dL / T + 1e-5
    exact, ties, bounded = check_against_oracle(acc, adv, nxt, gt, ol, Z, U, G, T, eps_q)
    parity_log.tokens(exact, ties)
    parity_log.count("sampled_draws_within_fp32_bound", bounded)
    # The logits form on the kernel's own logits meets the same bar.
    la, lad, ln = logits_verify_gpu(toks, logits, Zd, Ud, Gd, T)
    check_against_oracle(la, lad, ln, gt, ol, Z, U, G, T, eps_q)
    agree = int(np.sum((la == acc) & (ln == nxt)))
    parity_log.count("head_form_agrees_with_logits_form", agree)
    assert agree >= bs - ties - bounded
    if spread <= 0.05:
        assert np.any(acc == P) or bs < 8  # some requests accept the whole block


def test_verify_sampled_head_is_reusable_and_batches_beyond_64():
    """Two calls in a row on one workspace give the same results (the keys and
    arrival counters are left at zero); batch 70 takes two request windows."""
    bs, T = 70, 1.0
    case = make(small_bf16_cfg(batch=bs, temperature=T), 71, strong_coupling=True)
    gc = GpuCase(case)
    P, V = gc.P, gc.V
    L, Ph = gc.base()
    # Batch 70 has no statistics chain: build u and lse from the oracle's
    # forced chain on the GPU's own drafted tokens (the logits chain's).
    toks, logits = gc.chain(L, Ph, T, want_logits=True)
    torch.cuda.synchronize()
    gt = toks.cpu().numpy()
    ot, om, ol, ou, olse = oracle_forced(case, gt, T)
    seed = 72
    Z = (np.concatenate([ol.astype(np.float32), synth.normal((bs, 1, V), 1.0, seed, 1)], axis=1) +
         synth.normal((bs, P + 1, V), 1.0, seed, 2)).astype(np.float32)
    U = synth.uniform_open01((bs, P), seed, 3).astype(np.float32)
    G = synth.gumbel_noise((bs, V), seed + 2)
    Zd, Ud, Gd = to_dev(Z), to_dev(U), to_dev(G)
    u = to_dev(ou.astype(np.float32))
    lse = to_dev(olse.astype(np.float32))
    ws = B.workspace(B.domino_verify_sampled_head_workspace_bytes(bs, P))
    r1 = head_verify_gpu(gc, toks, L, u, lse, Zd, Ud, Gd, T, ws)
    r2 = head_verify_gpu(gc, toks, L, u, lse, Zd, Ud, Gd, T, ws)
    for a, b in zip(r1, r2):
        assert np.array_equal(a, b)
    assert np.any(r1[0] < P)  # some rejections: the residual kernel ran
    exact, ties, bounded = check_against_oracle(*r1, gt, ol, Z, U, G, T, 1e-4)
    parity_log.tokens(exact, ties)


def test_graph_captured_stats_step_matches_eager():
    """Base pass + statistics chain + head-form verification captured as one
    CUDA graph (the benchmark's sampled step at batch >= 5) gives the eager
    results bit for bit."""
    from draft_head_gb300.runtime import DominoDrafter
    from tests.test_gpu_next import _capture
    bs, T = 16, 1.0
    case = make(small_bf16_cfg(batch=bs, temperature=T), 81, strong_coupling=True)
    w = {k: to_dev(case[k]) for k in ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2")}
    P, V = case["P"], case["V"]
    dr = DominoDrafter(w, bs, P)
    assert dr.stats_supported()
    H = to_dev(case["H"])
    anchor = to_dev(case["anchor"].astype(np.int32))
    gm = to_dev(case["gumbel"])
    Z = to_dev((synth.normal((bs, P + 1, V), 1.0, 82, 0)).astype(np.float32))
    U = to_dev(synth.uniform_open01((bs, P), 82, 1).astype(np.float32))
    G = to_dev(synth.gumbel_noise((bs, V), 83))

    def step():
        dr.base(H)
        dr.chain_stats(anchor, T, gm[:, 1:, :], (P + 1) * V)
        dr.verify_sampled_head(Z, U, G, T)

    step()
    torch.cuda.synchronize()
    outs = lambda: (dr.tokens, dr.u_stats, dr.lse_stats, dr.accept, dr.advanced, dr.next_token)
    eager = [x.clone() for x in outs()]
    g = _capture(step)
    for x in (dr.tokens, dr.accept, dr.next_token):
        x.fill_(-7)
    dr.lse_stats.fill_(0.0)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs(), eager):
        assert torch.equal(a, b)
    assert dr.last_status() == 0
