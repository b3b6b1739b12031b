"""Small drafting cases run through whichever library the binding loaded
(libdomino.so, or libdomino_checked.so with DOMINO_LIB=checked): a chain at
batch 1 and 3 (greedy and Gumbel), the batched chain at batch 20, a tree, and
at batch 20 the statistics chain with the head-form sampled verification.
run() returns every output as nested lists plus the final status, so two
libraries can be compared bit for bit. `python -m tests.checked_cases` prints
them as one JSON line."""
from __future__ import annotations

import json

import numpy as np
import torch


def run() -> dict:
    from draft_head_gb300 import binding as B
    from tests.gpu_harness import GpuCase, make, small_bf16_cfg

    out = {}
    for bs, T in ((1, 0.0), (3, 1.0), (20, 0.0)):
        case = make(small_bf16_cfg(d=328, e=328, batch=bs, temperature=T), 500 + bs, strong_coupling=True)
        gc = GpuCase(case, n_nodes=12, top_m=16)
        L, Ph = gc.base()
        toks, lo = gc.chain(L, Ph, temperature=T, want_logits=True)
        out[f"chain{bs}_tokens"] = toks.cpu().numpy().tolist()
        out[f"chain{bs}_logits_sum"] = float(lo.double().sum().item())
        tok = torch.empty(bs, 13, dtype=torch.int32, device="cuda")
        par, dep = torch.empty_like(tok), torch.empty_like(tok)
        sco = torch.empty(bs, 13, dtype=torch.float32, device="cuda")
        B.dominotree_build(gc.head, L, Ph, gc.anchor, bs, case["P"], 12, 16, tok, par, dep, sco, gc.ws)
        out[f"tree{bs}"] = [tok.cpu().numpy().tolist(), par.cpu().numpy().tolist(), sco.cpu().numpy().tolist()]
        out[f"status{bs}"] = gc.status()
    # The statistics chain (batched, T = 1) and the head-form verification.
    from draft_head_gb300 import synth
    bs, T = 20, 1.0
    case = make(small_bf16_cfg(d=328, e=328, batch=bs, temperature=T), 540, strong_coupling=True)
    gc = GpuCase(case)
    P, V = case["P"], case["V"]
    L, Ph = gc.base()
    toks = torch.empty(bs, P, dtype=torch.int32, device="cuda")
    u = torch.empty(bs, P, gc.r, dtype=torch.float32, device="cuda")
    lse = torch.empty(bs, P, dtype=torch.float32, device="cuda")
    B.domino_draft_chain_stats(gc.head, L, Ph, gc.anchor, bs, P, T, gc.gumbel[:, 1:, :], (P + 1) * V, None, toks, u,
                               lse, gc.ws)
    Z = torch.from_numpy(synth.normal((bs, P + 1, V), 1.0, 541, 0).astype(np.float32)).cuda()
    U = torch.from_numpy(synth.uniform_open01((bs, P), 541, 1).astype(np.float32)).cuda()
    G = torch.from_numpy(synth.gumbel_noise((bs, V), 542)).cuda()
    acc = torch.empty(bs, dtype=torch.int32, device="cuda")
    adv, nxt = torch.empty_like(acc), torch.empty_like(acc)
    ws = B.workspace(B.domino_verify_sampled_head_workspace_bytes(bs, P))
    B.domino_verify_sampled_head(gc.head, toks, L, u, lse, Z, U, G, bs, P, T, acc, adv, nxt, ws)
    out["stats_tokens"] = toks.cpu().numpy().tolist()
    out["stats_lse"] = lse.cpu().numpy().tolist()
    out["stats_u_sum"] = float(u.double().sum().item())
    out["verify_head"] = [acc.cpu().numpy().tolist(), nxt.cpu().numpy().tolist()]
    out["status_stats_chain"] = gc.status()
    out["status_stats_verify"] = B.domino_last_status(ws)
    torch.cuda.synchronize()
    return out


if __name__ == "__main__":
    print(json.dumps(run()))
