"""The allocation-free chain entry point, checked against the regular one.

Some callers of this library cannot allocate device memory on their own: a
serving framework whose memory pool hands out no raw blocks, or a decode loop
that must not allocate once it has been warmed up. They call
domino_draft_chain_noalloc, which keeps its scratch in a fixed array inside
the library instead of a caller-provided workspace. These tests check, through
the C ABI, that it drafts the same tokens and corrected logits as
domino_draft_chain with a workspace, on two calls in a row (the second call
starts from whatever the first one left in the shared array), and that it
refuses sizes beyond its fixed limits.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from draft_head_gb300 import synth

if torch.cuda.is_available():
    from draft_head_gb300 import binding as B
    from tests.gpu_harness import GpuCase, make, small_bf16_cfg


# bf16 at rank 256 runs the small-batch kernel; fp32 heads and other ranks run
# the generic chain kernel, whose scratch (double-buffered accumulators, the
# global u rows) sits elsewhere in the fixed array.
@pytest.mark.parametrize("kind,bs,temperature", [("bf16", 1, 0.0), ("bf16", 3, 1.0), ("f32", 1, 0.0),
                                                 ("f32", 4, 0.0), ("bf16_r128", 2, 1.0)])
def test_noalloc_chain_matches_workspace_chain(kind, bs, temperature):
    if kind == "f32":
        cfg = dict(synth.CONFIGS["tiny_f32"], batch=bs, temperature=temperature)
        case = make(cfg, synth.case_seed("tiny_f32", 40 + bs), strong_coupling=True)
    else:
        r = 128 if kind == "bf16_r128" else 256
        case = make(small_bf16_cfg(d=328, e=328, r=r, batch=bs, temperature=temperature), 70 + bs,
                    strong_coupling=True)
    gc = GpuCase(case)
    L, Ph = gc.base()
    ref_tok, ref_logits = gc.chain(L, Ph, temperature=temperature, want_logits=True)
    assert gc.status() == 0

    g, stride = None, 0
    if temperature > 0.0:
        g = gc.gumbel[:, 1:, :]
        stride = gc.gumbel.shape[1] * case["V"]
    for _ in range(2):
        tok = torch.full((bs, case["P"]), -7, dtype=torch.int32, device="cuda")
        logits = torch.full((bs, case["P"], case["V"]), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        B.domino_draft_chain_noalloc(gc.head, L, Ph, gc.anchor, bs, case["P"], temperature, g, stride,
                                     None, tok, logits, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # Same kernel, same inputs, deterministic sums: bit-identical results.
        assert torch.equal(tok, ref_tok)
        assert torch.equal(logits, ref_logits)


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    case = make(small_bf16_cfg(d=328, e=328, batch=5), 79)
    gc = GpuCase(case)
    L, Ph = gc.base()
    tok = torch.empty(5, case["P"], dtype=torch.int32, device="cuda")
    with pytest.raises(B.DominoError) as err:
        B.domino_draft_chain_noalloc(gc.head, L, Ph, gc.anchor, 5, case["P"], 0.0, None, 0, None, tok, None)
    assert err.value.status == 2  # DOMINO_ERR_UNSUPPORTED
