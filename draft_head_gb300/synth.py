"""Seeded synthetic inputs for the Domino drafting hot path.

This module only draws random numbers and converts number formats. It holds
none of the method's arithmetic, so both the CUDA path and the CPU oracle can
take their inputs from it without sharing any computation.

Workloads (shapes follow the pages' Qwen3-4B / Qwen3-8B targets with block 16,
GRU hidden 1024 and bottleneck rank 256 -- "Domino: Decoupling Causal Modeling
from Autoregressive Drafting in Speculative Decoding Review", section 4-2
"Training strategy" table):

    tiny_f32         d=64,   V=1000,   g=32,   e=64,   r=16,  block 4,  batch 1,  fp32
    qwen3_4b_bs1     d=2560, V=151936, g=1024, e=2560, r=256, block 16, batch 1,  bf16, greedy
    qwen3_4b_bs64    as above, batch 64, Gumbel-max sampling at T=1
    qwen3_8b_bs32    d=e=4096, batch 32, greedy, targets match the draft w.p. 0.85
    qwen3_4b_tree    batch 16, best-first tree of 16 nodes, top-64 candidates

Value distributions: every head weight and the embedding ~ N(0, 0.02); the
backbone hidden states H ~ N(0, 1); the frozen LM head W_lm ~ N(0, 1/sqrt(d)),
so base logits are roughly N(0, 1). Draws are fp32 and, for the bf16
workloads, rounded to bf16 with round-to-nearest-even. Random streams are
split into fixed-size chunks, each with its own PCG64 generator keyed by
(seed, tensor id, chunk index), so the bytes do not depend on thread count.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 22

# Tensor ids for the random streams (fixed order: H, W_lm, emb, w_ih, w_hh,
# b_ih, b_hh, W1, W2, anchor, gumbel, target).
_TID = {"H": 0, "w_lm": 1, "emb": 2, "w_ih": 3, "w_hh": 4, "b_ih": 5, "b_hh": 6,
        "w1": 7, "w2": 8, "anchor": 9, "gumbel": 10, "target": 11, "tree_target": 12}

CONFIGS = {
    "tiny_f32": dict(index=1, dtype="f32", d=64, V=1000, g=32, e=64, r=16, block=4,
                     batch=1, temperature=0.0, target=("uniform", None), seeds=20),
    "qwen3_4b_bs1": dict(index=2, dtype="bf16", d=2560, V=151936, g=1024, e=2560, r=256,
                         block=16, batch=1, temperature=0.0, target=("flip", 0.2)),
    "qwen3_4b_bs64": dict(index=3, dtype="bf16", d=2560, V=151936, g=1024, e=2560, r=256,
                          block=16, batch=64, temperature=1.0, target=("flip", 0.2)),
    "qwen3_8b_bs32": dict(index=4, dtype="bf16", d=4096, V=151936, g=1024, e=4096, r=256,
                          block=16, batch=32, temperature=0.0, target=("match", 0.85)),
    "qwen3_4b_tree": dict(index=5, dtype="bf16", d=2560, V=151936, g=1024, e=2560, r=256,
                          block=16, batch=16, temperature=0.0, target=("flip", 0.2),
                          tree_nodes=16, top_m=64),
}


def case_seed(cfg_name: str, s: int) -> int:
    """Seed of sample s of a workload: 1000 * workload index + s."""
    return 1000 * CONFIGS[cfg_name]["index"] + s


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    flat_u = u.reshape(-1)
    flat_o = out.reshape(-1)
    for s in range(0, flat_u.size, _CHUNK):
        c = flat_u[s:s + _CHUNK]
        flat_o[s:s + _CHUNK] = ((c + (((c >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _gen(seed: int, tid: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(tid, chunk))))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal(shape, std: float, seed: int, tid: int) -> np.ndarray:
    """fp32 N(0, std^2) draws, filled chunk by chunk (thread-count independent)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    starts = list(range(0, n, _CHUNK))

    def fill(ci_s):
        ci, s = ci_s
        e = min(n, s + _CHUNK)
        _gen(seed, tid, ci).standard_normal(e - s, dtype=np.float32, out=out[s:e])
        out[s:e] *= np.float32(std)

    if len(starts) > 1:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, enumerate(starts)))
    else:
        for it in enumerate(starts):
            fill(it)
    return out.reshape(shape)


def uniform_open01(shape, seed: int, tid: int) -> np.ndarray:
    """fp64 uniform draws on the open interval (0, 1): (k + 1/2) / 2^24, k uniform."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    for ci, s in enumerate(range(0, n, _CHUNK)):
        e = min(n, s + _CHUNK)
        k = _gen(seed, tid, ci).integers(0, 1 << 24, size=e - s, dtype=np.int64)
        out[s:e] = (k.astype(np.float64) + 0.5) * (1.0 / (1 << 24))
    return out.reshape(shape)


def gumbel_noise(shape, seed: int) -> np.ndarray:
    """Standard Gumbel noise g = -log(-log U), U uniform on (0, 1), stored fp32.

    This is the random input of Gumbel-max sampling; both sides receive the
    same fp32 tensor."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    flat = out
    for ci, s in enumerate(range(0, n, _CHUNK)):
        e = min(n, s + _CHUNK)
        k = _gen(seed, _TID["gumbel"], ci).integers(0, 1 << 24, size=e - s, dtype=np.int64)
        u = (k.astype(np.float64) + 0.5) * (1.0 / (1 << 24))
        flat[s:e] = (-np.log(-np.log(u))).astype(np.float32)
    return out.reshape(shape)


def make_case(cfg: dict, seed: int, *, strong_coupling: bool = False,
              w2_zero: bool = False, batch: int | None = None,
              gumbel: bool | None = None) -> dict:
    """Draw one workload sample.

    Returns a dict with the dims and, per tensor, the stored representation:
    uint16 bf16 bits for the bf16 workloads, fp32 otherwise. Keys:
      H [batch, P, d], w_lm [V, d], emb [V, e], w_ih [3g, e], w_hh [3g, g],
      b_ih [3g], b_hh [3g], w1 [r, d+g], w2 [V, r], anchor [batch] int32,
      gumbel [batch, block, V] fp32 (row 0 unused) or None.
    strong_coupling: GRU weights and the S-columns of W1 drawn with std 0.2
    instead of 0.02, so that the state visibly moves the logits.
    w2_zero: W2 = 0 (the head-off ablation).
    """
    d, V, g, e, r = cfg["d"], cfg["V"], cfg["g"], cfg["e"], cfg["r"]
    B = cfg["block"]
    P = B - 1
    bs = cfg["batch"] if batch is None else batch
    bf16 = cfg["dtype"] == "bf16"
    ws = 0.2 if strong_coupling else 0.02

    def store(x):
        return f32_to_bf16_bits(x) if bf16 else np.ascontiguousarray(x, dtype=np.float32)

    out = dict(d=d, V=V, g=g, e=e, r=r, block=B, P=P, batch=bs, dtype=cfg["dtype"], seed=seed)
    out["H"] = store(normal((bs, P, d), 1.0, seed, _TID["H"]))
    out["w_lm"] = store(normal((V, d), 1.0 / np.sqrt(d), seed, _TID["w_lm"]))
    out["emb"] = store(normal((V, e), 0.02, seed, _TID["emb"]))
    out["w_ih"] = store(normal((3 * g, e), ws, seed, _TID["w_ih"]))
    out["w_hh"] = store(normal((3 * g, g), ws, seed, _TID["w_hh"]))
    out["b_ih"] = store(normal((3 * g,), 0.02, seed, _TID["b_ih"]))
    out["b_hh"] = store(normal((3 * g,), 0.02, seed, _TID["b_hh"]))
    w1 = normal((r, d + g), 0.02, seed, _TID["w1"])
    if strong_coupling:
        w1[:, d:] *= np.float32(10.0)
    out["w1"] = store(w1)
    w2 = normal((V, r), 0.02, seed, _TID["w2"])
    if w2_zero:
        w2[:] = 0.0
    out["w2"] = store(w2)
    out["anchor"] = _gen(seed, _TID["anchor"], 0).integers(0, V, size=bs).astype(np.int32)
    use_g = (cfg.get("temperature", 0.0) > 0.0) if gumbel is None else gumbel
    out["gumbel"] = gumbel_noise((bs, B, V), seed) if use_g else None
    out["temperature"] = float(cfg.get("temperature", 0.0)) if use_g else 0.0
    return out


def as_f32(x: np.ndarray) -> np.ndarray:
    """Stored tensor (bf16 bits or fp32) as fp32 values."""
    if x.dtype == np.uint16:
        return bf16_bits_to_f32(x)
    return np.asarray(x, dtype=np.float32)


def make_targets(draft: np.ndarray, mode: str, p, V: int, seed: int) -> np.ndarray:
    """Synthetic target tokens for verification.

    mode "uniform": iid uniform tokens.
    mode "flip":    keep each draft token with prob 1-p, else a uniform token != draft.
    mode "match":   keep each draft token with prob p, else a uniform token != draft.
    """
    rng = _gen(seed, _TID["target"], 0)
    draft = np.asarray(draft, dtype=np.int64)
    if mode == "uniform":
        return rng.integers(0, V, size=draft.shape).astype(np.int32)
    keep_p = (1.0 - p) if mode == "flip" else p
    keep = rng.random(draft.shape) < keep_p
    other = rng.integers(0, V - 1, size=draft.shape)
    other = other + (other >= draft)  # uniform over tokens != draft
    return np.where(keep, draft, other).astype(np.int32)


def make_tree_targets(node_token: np.ndarray, node_parent: np.ndarray, p: float, V: int, seed: int) -> np.ndarray:
    """Synthetic target next-tokens for a drafted tree, one per node slot [batch, N+1].

    At each node that has children, with prob 1-p the target's next token is the
    token of its first child (the first one popped), else a uniform token that is
    none of its children's tokens (the first child's if every token is a child);
    at a leaf it is uniform. Empty slots get -1.
    """
    tok = np.asarray(node_token, dtype=np.int64)
    par = np.asarray(node_parent, dtype=np.int64)
    bs, n1 = tok.shape
    rng = _gen(seed, _TID["tree_target"], 0)
    keep = rng.random((bs, n1)) >= p
    draw = rng.integers(0, V, size=(bs, n1, 4))  # rejection draws for "none of the children"
    out = np.full((bs, n1), -1, dtype=np.int32)
    for b in range(bs):
        for n in range(n1):
            if tok[b, n] < 0:
                continue
            kids = [int(tok[b, c]) for c in range(1, n1) if tok[b, c] >= 0 and par[b, c] == n]
            if kids and keep[b, n]:
                out[b, n] = kids[0]
                continue
            cand = [int(x) for x in draw[b, n] if int(x) not in kids]
            if not cand:
                cand = [t for t in range(V) if t not in kids] or kids  # every token a child: take one
            out[b, n] = cand[0]
    return out
