"""Helpers for the GPU parity tests: upload a seeded case, run the library's
entry points through the C ABI, and compare with the oracle under the
tolerances of the parity bar.

Tolerances (per the workload spec): logits max-abs 1e-4 on the fp32 path and
2e-2 on the bf16 path (bf16 operands, fp32 accumulation); tokens, accept
lengths and tree structure bit-exact, except where the oracle's own decision
margin is below 1e-3 (a near tie), which is counted and reported.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.domino_oracle as O
from draft_head_gb300 import binding as B
from draft_head_gb300 import synth
from tests import parity_log
from tests.tree_check import NEAR_TIE, compare_tree, compare_trees  # noqa: F401
TOL = {"f32": 1e-4, "bf16": 2e-2}
assert NEAR_TIE == 1e-3


def to_dev(x, dev="cuda"):
    if x is None:
        return None
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


class GpuCase:
    """Device copies of one case plus a prepared head and workspace."""

    def __init__(self, case: dict, n_nodes: int = 0, top_m: int = 0):
        self.case = case
        self.bs, self.P, self.V, self.r = case["batch"], case["P"], case["V"], case["r"]
        t = {k: to_dev(case[k]) for k in ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2", "H")}
        self.t = t
        self.head = B.Head(t["w_lm"], t["emb"], t["w_ih"], t["w_hh"], t["b_ih"], t["b_hh"], t["w1"], t["w2"])
        g = case["g"]
        self.table = torch.empty(case["V"] * 3 * g, dtype=torch.float32, device="cuda")
        self.ws = B.workspace(B.domino_workspace_bytes(self.head, self.bs, self.P, n_nodes, top_m))
        B.domino_prepare_gate_table(self.head, self.table, self.ws)
        self.head.set_gate_table(self.table)
        self.anchor = to_dev(case["anchor"].astype(np.int32))
        self.gumbel = to_dev(case["gumbel"]) if case.get("gumbel") is not None else None

    def base(self):
        L = torch.empty(self.bs, self.P, self.V, dtype=torch.float32, device="cuda")
        Ph = torch.empty(self.bs, self.P, self.r, dtype=torch.float32, device="cuda")
        B.domino_base_logits(self.head, self.t["H"], self.bs, self.P, L, Ph, self.ws)
        return L, Ph

    def chain(self, L, Ph, temperature=0.0, force=None, want_logits=False):
        toks = torch.empty(self.bs, self.P, dtype=torch.int32, device="cuda")
        lo = torch.empty(self.bs, self.P, self.V, dtype=torch.float32, device="cuda") if want_logits else None
        g = None
        stride = 0
        if temperature > 0.0:
            g = self.gumbel[:, 1:, :]  # drafted rows of the [batch, block, V] noise
            stride = self.gumbel.shape[1] * self.V
        f = to_dev(np.asarray(force, dtype=np.int32)) if force is not None else None
        B.domino_draft_chain(self.head, L, Ph, self.anchor, self.bs, self.P, temperature, g, stride, f, toks,
                             lo, self.ws)
        return toks, lo

    def status(self):
        return B.domino_last_status(self.ws)


def oracle_all(case, temperature=0.0, force=None, want_logits=True, requests=None):
    head = O.prepare_head(case)
    L = O.base_logits(case["H"], case["w_lm"]) if requests is None else None
    if requests is not None:
        L = np.full((case["batch"], case["P"], case["V"]), np.nan)
        for b in requests:
            L[b] = O.base_logits(case["H"][b], case["w_lm"])
    G = case["gumbel"][:, 1:, :] if temperature > 0.0 else None
    toks, margins, logits = O.draft_chain(head, case["H"], L, case["anchor"], temperature=temperature,
                                          gumbel=G, force=force, want_logits=want_logits, requests=requests)
    return head, L, toks, margins, logits


def gpu_candidates(L, M):
    """The candidate sets C_t the GPU selects from its own L_base [batch, P, V]
    (domino_topm_select, the select the tree build runs): [batch, P, M] ids."""
    bs, P, V = L.shape
    ids = torch.empty(bs * P, M, dtype=torch.int32, device=L.device)
    ws = B.workspace(B.domino_topm_workspace_bytes(bs * P, V, M))
    B.domino_topm_select(L.reshape(bs * P, V), bs * P, V, M, ids, None, ws)
    return ids.view(bs, P, M).cpu().numpy()


def compare_tokens(gpu_toks, ora_toks, margins, requests=None):
    """Free-running chains: equal up to each request's first divergence, and a
    divergence is only allowed at an oracle near tie. Returns (compared, near_ties)."""
    gpu_toks = np.asarray(gpu_toks)
    compared = 0
    ties = 0
    rows = range(gpu_toks.shape[0]) if requests is None else requests
    for b in rows:
        for i in range(gpu_toks.shape[1]):
            if gpu_toks[b, i] != ora_toks[b, i]:
                assert margins[b, i] < NEAR_TIE, (
                    f"token mismatch b={b} i={i}: gpu {gpu_toks[b, i]} oracle {ora_toks[b, i]} "
                    f"margin {margins[b, i]:.3g}")
                ties += 1
                break
            compared += 1
    parity_log.tokens(compared, ties)
    return compared, ties


def compare_forced(gpu_toks, ora_toks, margins, requests=None):
    """Teacher-forced chains: every position is compared; mismatches only at near ties."""
    gpu_toks = np.asarray(gpu_toks)
    rows = range(gpu_toks.shape[0]) if requests is None else requests
    ties = 0
    for b in rows:
        for i in range(gpu_toks.shape[1]):
            if gpu_toks[b, i] != ora_toks[b, i]:
                assert margins[b, i] < NEAR_TIE, f"forced mismatch b={b} i={i} margin {margins[b, i]:.3g}"
                ties += 1
    parity_log.tokens(gpu_toks.shape[1] * len(rows) - ties, ties)
    return ties


def check_logits(got, want, kind):
    """Max-abs logit error against the oracle within the parity bar; logged."""
    err = float(np.max(np.abs(np.asarray(got, dtype=np.float64) - want)))
    parity_log.logits(kind, err)
    assert err < TOL[kind], f"logits max-abs {err:.3g} above {TOL[kind]}"
    return err


def small_bf16_cfg(**over):
    """bf16 shapes small enough for a full oracle but spanning several tiles with
    ragged tails: V = 1000 (7 full 128-row tiles + 104), d = 320 (5 K-chunks)."""
    c = dict(index=90, dtype="bf16", d=320, V=1000, g=64, e=320, r=256, block=16, batch=1,
             temperature=0.0)
    c.update(over)
    return c


def make(cfg, seed, **kw):
    return synth.make_case(cfg, seed, **kw)


# Relative error of the kernel's fp32 p_v and q_v: each is exp2 of a
# pre-scaled value minus a log-sum-exp accumulated in fp32 over at most 151936
# terms, so a few ulps of a value near log2(V) ~ 17 (2^-19 each) plus the sum's
# rounding; 1e-5 is a generous bound.
_EPS_PQ = 1e-5


def _draw_within_fp32_error(Lb, Zb, Gb, j, tok_oracle, tok_gpu, T, eps_q=None):
    """The draw argmax_v log r_v + G_v at the rejection row j (r = max(p - q, 0),
    or p after all P accepted): true if the GPU's token scores within the fp32
    error of both candidates' log r_v of the oracle's token. log r_v's error is
    (|dp_v| + |dq_v|) / r_v <= _EPS_PQ (p_v + q_v) / r_v, which grows without
    bound where p and q almost cancel; the 1e-3 margin bar alone cannot cover
    those draws, so they are counted separately. eps_q replaces _EPS_PQ for q
    where the kernel's draft logits themselves differ from the oracle's (the
    head form rebuilds them): |dq_v| / q_v <= |dL| / T + _EPS_PQ."""
    P = Lb.shape[0]
    p = O._softmax64(np.asarray(Zb[j], np.float64) / T)
    q = O._softmax64(np.asarray(Lb[j], np.float64) / T) if j < P else np.zeros_like(p)
    r = np.maximum(p - q, 0.0)
    if not np.any(r > 0):
        r, q = p, np.zeros_like(p)
    if r[tok_gpu] <= 0.0:
        return False
    score = lambda v: np.log(r[v]) + float(Gb[v])
    eq = _EPS_PQ if eps_q is None else eps_q
    err = lambda v: (_EPS_PQ * p[v] + eq * q[v]) / r[v]
    return score(tok_oracle) - score(tok_gpu) <= err(tok_oracle) + err(tok_gpu)
