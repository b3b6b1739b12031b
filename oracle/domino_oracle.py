"""CPU oracle for the Domino drafting hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this module. The product path (the CUDA library and its binding) never calls
it, and it shares no code with that path: it imports numpy only.

It is a plain, slow, fp64 restatement of what the pages define. Sources, by
page title (abbreviation in brackets):

  [Review]  "Domino: Decoupling Causal Modeling from Autoregressive Drafting in
            Speculative Decoding Review" (dimensionstp.github.io)
  [NL]      "Technische Samenvatting: Domino" (gist.science, Dutch)
  [News]    "上交大突破：多米诺推理策略实现AI推理速度近6倍能力提升" (163.com)
  [Tree]    "DominoTree: Conditional Tree-Structured Drafting with Domino for
            Speculative Decoding" (gist.science, Chinese)

Readings where the pages are silent:
  R1  GRU cell = the standard gated recurrent unit with separate input and
      hidden biases and the reset gate applied to (W_hn h + b_hn); gate order
      r, z, n in the stacked weight rows.
  R2  S_{-1} = 0; the anchor token (block position 0) is the first GRU input.
  R3  A block of B positions holds the anchor plus P = B - 1 drafted positions;
      all arrays with a position axis hold the P drafted rows, row i being
      block position i + 1.
  R4  The concatenation [H_i ; S_{i-1}] puts H first (W1 columns [0, d) act on
      H, columns [d, d + g) on S).
  R5  No bias in W1 or W2.
  R9  argmax ties go to the lowest token id.
  R10 Sampling at temperature T > 0 is Gumbel-max: argmax(L / T + G) with the
      noise G supplied as an input.
  R12 Tokens advanced per cycle = accepted length + 1 (the target's own token).
  Decision precision: every value that decides an integer (an argmax, a
  top-M membership, a heap order) is rounded to fp32 first, the precision of
  the GPU kernels; the arithmetic before that point is fp64.
  T1..T10 (tree): see tree_build.  V1..V3 (tree acceptance): see tree_verify.
  S1..S4 (verification at T > 0): see verify_stochastic; S6 (the draft-side
  statistics that stand in for the logits): see draft_chain_stats.

Nothing here is pinned only against itself: tests/test_oracle_pins.py checks it
against hand-worked values, library routines (torch.nn.GRUCell, scipy),
closed forms, brute-force enumeration and invariants.
"""
from __future__ import annotations

import heapq

import numpy as np

__all__ = [
    "widen", "prepare_head", "base_logits", "sigmoid", "silu", "gru_cell",
    "draft_chain", "verify", "top_m", "tree_build", "head_param_count",
    "tree_verify", "draft_chain_headoff", "tree_build_marginal", "verify_stochastic",
    "draft_chain_stats",
]

_ROWS = 8192  # rows of a big weight converted to fp64 at a time


def widen(x) -> np.ndarray:
    """Any stored tensor (fp32 values, or uint16 bf16 bits) as fp64 values."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def prepare_head(case: dict) -> dict:
    """fp64 copies of the small head weights; W_lm and emb stay as stored and
    are widened a block of rows at a time."""
    return dict(
        d=case["d"], e=case["e"], g=case["g"], r=case["r"], V=case["V"],
        w_lm=case["w_lm"], emb=case["emb"],
        w_ih=widen(case["w_ih"]), w_hh=widen(case["w_hh"]),
        b_ih=widen(case["b_ih"]), b_hh=widen(case["b_hh"]),
        w1=widen(case["w1"]), w2=widen(case["w2"]),
    )


def head_param_count(d: int, e: int, g: int, r: int, V: int, shared_embedding: bool = True) -> int:
    """Trainable parameters of the Domino head under readings R1/R5 and the
    shared target embedding: GRU (W_ih, W_hh, b_ih, b_hh), W1 [r, d+g], W2 [V, r]
    ([News] section 四 quotes the head as adding 56M parameters)."""
    gru = 3 * g * e + 3 * g * g + 2 * 3 * g
    n = gru + r * (d + g) + V * r
    if not shared_embedding:
        n += V * e
    return n


# ---------------------------------------------------------------------------
# a1: base logits.  [NL] "Parallel Draft-ruggengraat": the block's hidden
# states go through the frozen target LM head once: L_base_i = H_i . W_lm^T.
# ---------------------------------------------------------------------------
def base_logits(H, w_lm) -> np.ndarray:
    """L_base[..., v] = sum_k H[..., k] * W_lm[v, k] in fp64. H [..., d], W_lm [V, d]."""
    Hf = widen(H)
    lead = Hf.shape[:-1]
    H2 = Hf.reshape(-1, Hf.shape[-1])
    V = np.asarray(w_lm).shape[0]
    out = np.empty((H2.shape[0], V), dtype=np.float64)
    for s in range(0, V, _ROWS):
        out[:, s:s + _ROWS] = H2 @ widen(w_lm[s:s + _ROWS]).T
    return out.reshape(*lead, V)


def base_logit_entries(H, w_lm, rows, cols) -> np.ndarray:
    """Single entries L_base[row, col] (rows index the flattened [batch*P] axis),
    each a length-d dot product; for sampled checks at full size."""
    Hf = widen(H).reshape(-1, np.asarray(H).shape[-1])
    out = np.empty(len(rows), dtype=np.float64)
    for n, (i, v) in enumerate(zip(rows, cols)):
        out[n] = float(np.dot(Hf[i], widen(w_lm[v])))
    return out


# ---------------------------------------------------------------------------
# Activations.
# ---------------------------------------------------------------------------
def sigmoid(t):
    return 1.0 / (1.0 + np.exp(-t))


def silu(t):
    """SiLU(t) = t * sigmoid(t) = t / (1 + e^-t) ([News] section 四: the
    bottleneck goes through a SiLU activation)."""
    return t / (1.0 + np.exp(-t))


# ---------------------------------------------------------------------------
# a3: GRU causal encoder.  [News] section 四 and [NL] "Causale Encoder": a GRU
# with hidden size 1024 reads the embeddings of the drafted tokens in order;
# the gate equations are reading R1.
# ---------------------------------------------------------------------------
def gru_cell(x, h, w_ih, w_hh, b_ih, b_hh):
    """One GRU step. x [e], h [g] fp64; w_ih [3g, e], w_hh [3g, g] rows (r, z, n)."""
    g = h.shape[-1]
    gi = w_ih @ x + b_ih
    gh = w_hh @ h + b_hh
    r = sigmoid(gi[:g] + gh[:g])
    z = sigmoid(gi[g:2 * g] + gh[g:2 * g])
    n = np.tanh(gi[2 * g:] + r * gh[2 * g:])
    return (1.0 - z) * n + z * h


def _emb_row(head, tok) -> np.ndarray:
    return widen(np.asarray(head["emb"])[int(tok)])


def _gru_on_token(head, tok, h):
    return gru_cell(_emb_row(head, tok), h, head["w_ih"], head["w_hh"], head["b_ih"], head["b_hh"])


def _bottleneck(head, H_i, S):
    """u = SiLU(W1 . [H_i ; S]) ([NL] "Low-Rank Correctie-head"; readings R4, R5)."""
    x = np.concatenate([widen(H_i), S])
    return silu(head["w1"] @ x)


def _fp32_argmax(values_f64):
    """argmax of the fp32-rounded values, ties to the lowest id (R9); also the
    fp32 margin between the best and the second-best value."""
    v32 = np.asarray(values_f64, dtype=np.float64).astype(np.float32)
    best = int(np.argmax(v32))  # numpy returns the first maximal index
    if v32.size > 1:
        top2 = np.partition(v32.astype(np.float64), -2)[-2:]
        margin = float(top2[1] - top2[0])
    else:
        margin = float("inf")
    return best, margin


# ---------------------------------------------------------------------------
# a3..a5: the sequential chain.  [NL] "Domino-head": L_i = L_base_i + dL_i with
# dL_i = W2 SiLU(W1 [H_i ; S_{i-1}]); tokens are drawn from the corrected
# distribution.  [Review] section 3-2: the correction is added in logit space.
# ---------------------------------------------------------------------------
def draft_chain(head, H, L_base, anchor, temperature: float = 0.0, gumbel=None,
                force=None, want_logits: bool = False, requests=None):
    """Run the Domino head chain per request.

    H [batch, P, d]; L_base [batch, P, V] (fp64); anchor [batch];
    gumbel [batch, P, V] or None (row i is the noise of block position i+1);
    force [batch, P] or None: teacher-forced GRU inputs (the token fed to the GRU
    after position i is force[b, i] instead of the drafted one).
    requests: optional subset of batch indices to run (others are left -1/NaN).

    Returns (tokens [batch, P] int64, margins [batch, P] fp64, logits or None).
    """
    H = np.asarray(H)
    bs, P = H.shape[0], H.shape[1]
    V = head["V"]
    tokens = np.full((bs, P), -1, dtype=np.int64)
    margins = np.full((bs, P), np.nan)
    logits = np.full((bs, P, V), np.nan) if want_logits else None
    for b, i, _u, L, tok, margin in _chain_rows(head, H, L_base, anchor, temperature, gumbel, force, requests):
        if want_logits:
            logits[b, i] = L
        tokens[b, i], margins[b, i] = tok, margin
    return tokens, margins, logits


def _chain_rows(head, H, L_base, anchor, temperature, gumbel, force, requests):
    """The chain's steps in order: yields (b, i, u_i, L_i, token, margin) for
    every drafted row of the requests run (all when requests is None)."""
    bs, P = H.shape[0], H.shape[1]
    g = head["g"]
    todo = range(bs) if requests is None else requests
    for b in todo:
        S = _gru_on_token(head, anchor[b], np.zeros(g))  # S_0 (R2)
        for i in range(P):
            u = _bottleneck(head, H[b, i], S)
            L = np.asarray(L_base[b, i], dtype=np.float64) + head["w2"] @ u
            if temperature > 0.0:
                dec = L / temperature + np.asarray(gumbel[b, i], dtype=np.float64)
            else:
                dec = L
            tok, margin = _fp32_argmax(dec)
            yield b, i, u, L, tok, margin
            if i < P - 1:
                nxt = force[b, i] if force is not None else tok
                S = _gru_on_token(head, nxt, S)


def draft_chain_stats(head, H, L_base, anchor, temperature: float = 0.0, gumbel=None, force=None,
                      requests=None):
    """The chain with, per drafted row, what a verification at temperature T
    needs in place of the full corrected logits (reading S6): the bottleneck
    activations u_i (from which L_i = L_base_i + W2 u_i follows for any token)
    and the log-partition lse_i = logsumexp_v L_i[v] / T' of the draft
    distribution softmax(L_i / T'), T' = T for T > 0 and 1 at T = 0.

    Returns (tokens [batch, P], margins [batch, P], u [batch, P, r],
    lse [batch, P]), fp64 where real-valued."""
    H = np.asarray(H)
    bs, P = H.shape[0], H.shape[1]
    tau = float(temperature) if temperature > 0.0 else 1.0
    tokens = np.full((bs, P), -1, dtype=np.int64)
    margins = np.full((bs, P), np.nan)
    us = np.full((bs, P, head["r"]), np.nan)
    lse = np.full((bs, P), np.nan)
    for b, i, u, L, tok, margin in _chain_rows(head, H, L_base, anchor, temperature, gumbel, force, requests):
        tokens[b, i], margins[b, i] = tok, margin
        us[b, i] = u
        lse[b, i] = _logsumexp(L / tau)
    return tokens, margins, us, lse


# ---------------------------------------------------------------------------
# a6: longest accepted prefix.  [Review] section 1-1: the target verifies the
# draft block in one pass; A = tokens advanced per cycle (reading R12).
# ---------------------------------------------------------------------------
def verify(draft, target):
    """accept[b] = largest k with draft[b, :k] == target[b, :k]; advanced = accept + 1."""
    draft = np.asarray(draft)
    target = np.asarray(target)
    bs, P = draft.shape
    accept = np.zeros(bs, dtype=np.int64)
    for b in range(bs):
        k = 0
        while k < P and draft[b, k] == target[b, k]:
            k += 1
        accept[b] = k
    return accept, accept + 1


# ---------------------------------------------------------------------------
# a7: top-M candidate limit.  [Tree] "候选限制（Top-M）": the per-node
# correction is applied only to the M best marginal candidates at each depth.
# ---------------------------------------------------------------------------
def top_m(row_values, M: int):
    """Ids of the M largest fp32-rounded values, ordered by value desc then id
    asc; also the fp32 gap between the M-th and (M+1)-th value."""
    v32 = np.asarray(row_values, dtype=np.float64).astype(np.float32)
    ids = np.arange(v32.size)
    order = np.lexsort((ids, -v32.astype(np.float64)))
    sel = order[:M]
    gap = float(v32[order[M - 1]]) - float(v32[order[M]]) if v32.size > M else float("inf")
    return sel.astype(np.int64), gap


def _logsumexp(x):
    m = np.max(x)
    return m + np.log(np.sum(np.exp(x - m)))


# ---------------------------------------------------------------------------
# a8: DominoTree best-first expansion.  [Tree] "条件评分的最佳优先堆": a max
# priority queue keyed by cumulative path log-probability; children are scored
# with the Domino correction recomputed along the node's own path, H being
# shared by all paths; a fixed budget of nodes.
# Readings:
#  T1 root = anchor, node 0, depth 0, score 0, state S_0 = GRU(emb[anchor], 0);
#     the budget counts drafted nodes (root excluded).
#  T2 C_t = top-M of L_base[t] (block position t+1), shared by every node that
#     expands into depth t+1.
#  T3 child c of node n at depth t: l_c = L_base[t, c] + W2[c] . SiLU(W1 [H_t ; S_n]),
#     logp_c = l_c / T - logsumexp over C_t of l / T (normalised over the
#     M-slice; T = 1 when the workload decodes greedily).
#  T10 scoring temperature: [Tree] 实验结果 evaluates the tree at decoding
#     temperatures 0, 0.5 and 1. At T > 0 the children are ranked by the
#     draft's tempered log-probabilities log-softmax(l / T) over the slice;
#     at T = 0 (greedy decoding) by the draft's own log-softmax(l).
#  T4 score(child) = score(parent) + logp_c (in fp32, reading "decision precision").
#  T5 all M children are pushed.
#  T6 pop the largest score; ties -> smaller parent id, then smaller token id.
#  T7 node ids 1..N in pop order.
#  T8 S_node = GRU(emb[token], S_parent), computed when the node is expanded;
#     no expansion at depth P, none after the N-th pop.
#  T9 requests are independent.
# If the heap runs dry before N pops (tiny trees), the remaining node slots are
# token = parent = depth = -1, score = -inf.
# ---------------------------------------------------------------------------
def _score_temperature(temperature: float) -> float:
    """Reading T10: the temperature the tree's log-softmax uses."""
    if temperature < 0.0:
        raise ValueError("temperature must be >= 0")
    return 1.0 if temperature == 0.0 else float(temperature)


def tree_build(head, H, L_base, anchor, n_nodes: int, M: int, requests=None, temperature: float = 0.0):
    """Returns dict of node_token/node_parent/node_depth [batch, N+1] int64,
    node_score [batch, N+1] fp32, plus near-tie diagnostics:
    pop_margin [batch, N+1] (gap between the popped key and the next key),
    cand_gap [batch, P] (top-M boundary gap) and cands [batch, P, M] (the
    candidate ids C_t, -1 for requests not run)."""
    tau = _score_temperature(temperature)
    H = np.asarray(H)
    bs, P = H.shape[0], H.shape[1]
    g = head["g"]
    N = n_nodes
    tok = np.full((bs, N + 1), -1, dtype=np.int64)
    par = np.full((bs, N + 1), -1, dtype=np.int64)
    dep = np.full((bs, N + 1), -1, dtype=np.int64)
    sco = np.full((bs, N + 1), -np.inf, dtype=np.float32)
    pop_margin = np.full((bs, N + 1), np.inf)
    cand_gap = np.full((bs, P), np.inf)
    cand_ids = np.full((bs, P, M), -1, dtype=np.int64)
    todo = range(bs) if requests is None else requests
    for b in todo:
        cands = []
        for t in range(P):
            c, gap = top_m(L_base[b, t], M)
            cands.append(c)
            cand_gap[b, t] = gap
            cand_ids[b, t, :len(c)] = c
        states = {0: _gru_on_token(head, anchor[b], np.zeros(g))}
        tok[b, 0], par[b, 0], dep[b, 0], sco[b, 0] = anchor[b], -1, 0, np.float32(0.0)
        heap = []

        def expand(n):
            t = int(dep[b, n])
            if t >= P:
                return
            u = _bottleneck(head, H[b, t], states[n])
            C = cands[t]
            l = (np.asarray(L_base[b, t], dtype=np.float64)[C] + head["w2"][C] @ u) / tau
            logp = (l - _logsumexp(l)).astype(np.float32)
            for c, lp in zip(C, logp):
                s = np.float32(sco[b, n] + lp)
                heapq.heappush(heap, (-float(s), n, int(c), t + 1))

        expand(0)
        for k in range(1, N + 1):
            if not heap:
                break
            negs, p, c, t = heapq.heappop(heap)
            if heap:
                pop_margin[b, k] = heap[0][0] - negs
            tok[b, k], par[b, k], dep[b, k], sco[b, k] = c, p, t, np.float32(-negs)
            if k < N and t < P:
                states[k] = _gru_on_token(head, c, states[p])
                expand(k)
    return dict(node_token=tok, node_parent=par, node_depth=dep, node_score=sco,
                pop_margin=pop_margin, cand_gap=cand_gap, cands=cand_ids)


# ---------------------------------------------------------------------------
# Tree acceptance.  [Tree] "验证": the tree is verified with the standard
# tree-attention scheme of DDTree / SpecInfer, an ancestor-only causal mask,
# unchanged and lossless.  The target pass itself is not part of this path;
# its greedy next token after every node's root path is an input.
# Readings:
#  V1 target_next[b, n] = the target's greedy token after the root path of
#     node n (node 0 = the anchor); empty node slots (token -1) are ignored.
#  V2 the walk starts at the root; at node n it moves to the child whose token
#     equals target_next[n] (children of one node carry distinct tokens, so at
#     most one matches) and stops when no child matches.
#  V3 accept = depth of the last node reached, advanced = accept + 1 (the
#     target's own token after it, reading R12).
# The attention mask row of node i marks node i and its ancestors.
# ---------------------------------------------------------------------------
def tree_verify(node_token, node_parent, target_next):
    """node_token, node_parent, target_next [batch, N+1].  Returns
    (accept [batch], advanced [batch], path [batch, N+1] node ids of the
    accepted root path, -1 after its end, mask [batch, N+1, N+1] uint8)."""
    tok = np.asarray(node_token)
    par = np.asarray(node_parent)
    tgt = np.asarray(target_next)
    bs, n1 = tok.shape
    accept = np.zeros(bs, dtype=np.int64)
    path = np.full((bs, n1), -1, dtype=np.int64)
    mask = np.zeros((bs, n1, n1), dtype=np.uint8)
    for b in range(bs):
        for i in range(n1):
            if tok[b, i] < 0:
                continue
            j = i
            while j >= 0:
                mask[b, i, j] = 1
                j = par[b, j] if j > 0 else -1
        node, depth = 0, 0
        path[b, 0] = 0
        while True:
            nxt = -1
            for c in range(1, n1):
                if tok[b, c] >= 0 and par[b, c] == node and tok[b, c] == tgt[b, node]:
                    nxt = c
                    break
            if nxt < 0:
                break
            node, depth = nxt, depth + 1
            path[b, depth] = node
        accept[b] = depth
    return accept, accept + 1, path, mask


# ---------------------------------------------------------------------------
# The pages' ablation baselines with the correction head off.  [Review] and
# [News]: the parallel backbone alone drafts every position from its marginal
# logits (DFlash-style).  [Tree] "核心贡献" (ablation): the same best-first tree
# scored with path-independent marginal log-probabilities (DDTree-style).
# Both equal the full method with W2 = 0, which the pins check.
# ---------------------------------------------------------------------------
def draft_chain_headoff(L_base, temperature: float = 0.0, gumbel=None):
    """tokens[b, i] = argmax L_base[b, i] (T = 0) or argmax(L_base[b, i] / T + G[b, i]),
    decided in fp32, ties to the lowest id.  Returns (tokens, margins)."""
    L_base = np.asarray(L_base)
    bs, P = L_base.shape[0], L_base.shape[1]
    tokens = np.full((bs, P), -1, dtype=np.int64)
    margins = np.full((bs, P), np.nan)
    for b in range(bs):
        for i in range(P):
            L = np.asarray(L_base[b, i], dtype=np.float64)
            dec = L / temperature + np.asarray(gumbel[b, i], dtype=np.float64) if temperature > 0.0 else L
            tokens[b, i], margins[b, i] = _fp32_argmax(dec)
    return tokens, margins


def tree_build_marginal(L_base, anchor, n_nodes: int, M: int, temperature: float = 0.0):
    """Best-first tree (readings T1, T2, T4-T10) whose child log-probabilities
    are the marginal ones: logp_c = L_base[t, c] / T - logsumexp over C_t of
    L_base / T (T = 1 at temperature 0).  Same outputs as tree_build."""
    tau = _score_temperature(temperature)
    L_base = np.asarray(L_base)
    bs, P = L_base.shape[0], L_base.shape[1]
    N = n_nodes
    tok = np.full((bs, N + 1), -1, dtype=np.int64)
    par = np.full((bs, N + 1), -1, dtype=np.int64)
    dep = np.full((bs, N + 1), -1, dtype=np.int64)
    sco = np.full((bs, N + 1), -np.inf, dtype=np.float32)
    pop_margin = np.full((bs, N + 1), np.inf)
    cand_gap = np.full((bs, P), np.inf)
    cand_ids = np.full((bs, P, M), -1, dtype=np.int64)
    for b in range(bs):
        cands, logps = [], []
        for t in range(P):
            c, gap = top_m(L_base[b, t], M)
            l = np.asarray(L_base[b, t], dtype=np.float64)[c] / tau
            cands.append(c)
            logps.append((l - _logsumexp(l)).astype(np.float32))
            cand_gap[b, t] = gap
            cand_ids[b, t, :len(c)] = c
        tok[b, 0], par[b, 0], dep[b, 0], sco[b, 0] = anchor[b], -1, 0, np.float32(0.0)
        heap = []

        def expand(n):
            t = int(dep[b, n])
            if t >= P:
                return
            for c, lp in zip(cands[t], logps[t]):
                heapq.heappush(heap, (-float(np.float32(sco[b, n] + lp)), n, int(c), t + 1))

        expand(0)
        for k in range(1, N + 1):
            if not heap:
                break
            negs, p, c, t = heapq.heappop(heap)
            if heap:
                pop_margin[b, k] = heap[0][0] - negs
            tok[b, k], par[b, k], dep[b, k], sco[b, k] = c, p, t, np.float32(-negs)
            if k < N and t < P:
                expand(k)
    return dict(node_token=tok, node_parent=par, node_depth=dep, node_score=sco,
                pop_margin=pop_margin, cand_gap=cand_gap, cands=cand_ids)


# ---------------------------------------------------------------------------
# Verification at temperature T > 0.  The 163.com report (section 五 and the
# interface notes): drafts are checked by the standard speculative-decoding
# procedure and the output keeps the target's probabilities; the DominoTree
# page (实验结果, 无损性): lossless within floating-point rounding.
# Readings:
#  S1 draft distribution q_i = softmax(L_i / T) (what the Gumbel-max chain
#     samples from), target distribution p_i = softmax(Z_i / T); Z [batch,
#     P + 1, V] are the target's logits (synthetic here), row P the position
#     after the last drafted token.
#  S2 the standard scheme: accept x_i while U_i < p_i(x_i) / q_i(x_i); at the
#     first rejection j the next token is drawn from norm(max(0, p_j - q_j));
#     if all P are accepted it is drawn from p_P.
#  S3 the draw uses Gumbel-max over V with noise G [batch, V] supplied as an
#     input: argmax_v log r_v + G_v; if the residual is zero everywhere (p and
#     q equal in fp32) it is drawn from p_j instead.
#  S4 accept = j, advanced = j + 1 (reading R12).
# Decisions are taken in fp32 (the acceptance ratio and the argmax values are
# rounded to fp32 before comparing).
# ---------------------------------------------------------------------------
def _softmax64(z):
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z)
    e = np.exp(z - m)
    return e / np.sum(e)


def verify_stochastic(draft, draft_logits, target_logits, uniform, gumbel, temperature: float):
    """draft [batch, P] ids; draft_logits [batch, P, V]; target_logits
    [batch, P + 1, V]; uniform [batch, P] in (0, 1); gumbel [batch, V].
    Returns (accept [batch], advanced [batch], next_token [batch],
    ratio_margin [batch]: min over decided positions of |U - ratio| in fp32,
    token_margin [batch]: gap between the best and second-best draw scores)."""
    draft = np.asarray(draft)
    L = np.asarray(draft_logits)
    Z = np.asarray(target_logits)
    bs, P = draft.shape
    T = float(temperature)
    accept = np.zeros(bs, dtype=np.int64)
    nxt = np.zeros(bs, dtype=np.int64)
    rmargin = np.full(bs, np.inf)
    tmargin = np.full(bs, np.inf)
    for b in range(bs):
        j = P
        for i in range(P):
            x = int(draft[b, i])
            q = _softmax64(np.asarray(L[b, i], dtype=np.float64) / T)
            p = _softmax64(np.asarray(Z[b, i], dtype=np.float64) / T)
            ratio = np.float32(min(1.0, p[x] / q[x]) if q[x] > 0 else 1.0)
            u = np.float32(uniform[b, i])
            rmargin[b] = min(rmargin[b], abs(float(u) - float(ratio)))
            if not (u < ratio):
                j = i
                break
        p = _softmax64(np.asarray(Z[b, j], dtype=np.float64) / T)
        if j < P:
            q = _softmax64(np.asarray(L[b, j], dtype=np.float64) / T)
            r = np.maximum(p - q, 0.0)
            base = r if np.any(r > 0) else p
        else:
            base = p
        with np.errstate(divide="ignore"):
            score = np.log(base) + np.asarray(gumbel[b], dtype=np.float64)
        nxt[b], tmargin[b] = _fp32_argmax(score)
        accept[b] = j
    return accept, accept + 1, nxt, rmargin, tmargin
