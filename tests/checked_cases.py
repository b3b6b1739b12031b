"""Small drafting cases run through whichever library the binding loaded
(libdomino.so, or libdomino_checked.so with DOMINO_LIB=checked): a chain at
batch 1 and 3 (greedy and Gumbel), the batched chain at batch 20, and a tree.
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
    torch.cuda.synchronize()
    return out


if __name__ == "__main__":
    print(json.dumps(run()))
