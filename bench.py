#!/usr/bin/env python
"""Benchmark of the Domino drafting hot path on one GB300 per rank.

A step is one speculative drafting cycle over one batch of synthetic input:
base logits (+ the H-half of the bottleneck) for the whole block, the
sequential chain of GRU + low-rank correction + sampling, and verification of
the drafted block against synthetic target tokens. The default workload is
the Qwen3-4B shape at batch 1 (d 2560, vocabulary 151936, GRU 1024, rank 256,
block 16, greedy).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, same metric

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs its own
replica of the workload (weak scaling, no data-path collective); value is the
total over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "drafted tokens/s + chain latency (block16, Qwen3-4B shape); % HBM / TC roofline"
UNIT = "drafted tok/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="domino", choices=["domino", "reference"])
    ap.add_argument("--workload", default="qwen3_4b_bs1")
    ap.add_argument("--variant", default="domino", choices=["domino", "headoff"],
                    help="headoff: the correction head switched off (per-position argmax of the base "
                         "logits for chains, the marginal-scored tree for trees)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="report the eager launches as the headline instead of the step replayed as one "
                         "captured CUDA graph")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the headline workload only (by default, at one GPU, the batch-64, 8B batch-32 "
                         "and tree workloads follow it, reported under 'workloads')")
    ap.add_argument("--tree-temperature", type=float, default=0.0,
                    help="scoring temperature of the tree when the headline workload is a tree")
    return ap.parse_args()


def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of x over all ranks (the slowest replica's time)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job drafted tokens/s: every rank drafts the same amount; the job
    takes as long as its slowest rank."""
    return world * tokens_per_rank / (max_ms / 1e3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# --------------------------------------------------------------------------- peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# Source files that define each kernel (with the shared device header); a
# recorded DRAM-traffic figure holds only while these are unchanged.
KERNEL_SOURCES = {
    "gemm_bf16_tc": ["gemm.cu"],
    "chain_small_kernel": ["chain_small.cu"],
    "chain_batched_kernel": ["chain_batched.cu"],
    "chain_kernel": ["chain.cu"],
    "tree_kernel": ["tree.cu"],
    "topm + tree_kernel": ["tree.cu"],
    "headoff_chain_kernel": ["headoff.cu"],
    "topm + tree_marginal_kernel": ["tree.cu", "headoff.cu"],
}


def csrc_hash(kernel: str):
    h = hashlib.sha256()
    d = os.path.join(ROOT, "draft_head_gb300", "csrc")
    for f in KERNEL_SOURCES.get(kernel, []) + ["common.cuh"]:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def chain_kernel_name(cfg: dict, bs: int) -> str:
    """Which chain kernel the library picks for this shape (the dispatch rule of
    launch_chain: small-batch, batched tensor-core, or the generic kernel)."""
    if cfg["dtype"] == "bf16" and cfg["r"] == 256:
        if bs <= 4:
            return "chain_small_kernel"
        if bs <= 64 and cfg["g"] % 64 == 0 and cfg["V"] % 4 == 0:
            return "chain_batched_kernel"
    return "chain_kernel"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("csrc_hash") != csrc_hash(kernel):
        return None
    return float(e["dram_bytes_per_launch"])


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = [l for (t, l) in self.lines if t0 - 0.12 <= t <= t1 + 0.12] or [l for (_, l) in self.lines]
        for l in window:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- CPU oracle
def oracle_cycle_sample(case, vocab_rows: int, target, mode: str = "chain", tree=(0, 0)):
    """One cycle of the oracle on a vocabulary slice [0, vocab_rows) of one request:
    base pass, then the chain / head-off chain / tree / marginal tree, then acceptance.
    Returns drafted-unit equivalents processed (P or N, times vocab_rows / V)."""
    import oracle.domino_oracle as O
    V = case["V"]
    sub = dict(case)
    sub["V"] = vocab_rows
    sub["w_lm"] = case["w_lm"][:vocab_rows]
    sub["w2"] = case["w2"][:vocab_rows]
    head = O.prepare_head(sub)
    H = case["H"][:1]
    L = O.base_logits(H, sub["w_lm"])
    anchor = np.minimum(case["anchor"][:1], vocab_rows - 1)
    sub["emb"] = case["emb"]
    if mode in ("tree", "marginal"):
        N, M = tree[0], min(tree[1], vocab_rows)
        tr = (O.tree_build(head, H, L, anchor, N, M) if mode == "tree"
              else O.tree_build_marginal(L, anchor, N, M))
        tnext = np.minimum(np.resize(target[:1], (1, N + 1)), vocab_rows - 1)
        O.tree_verify(tr["node_token"], tr["node_parent"], tnext)
        return N * vocab_rows / V
    if mode == "headoff":
        toks, _ = O.draft_chain_headoff(L)
    else:
        toks, _, _ = O.draft_chain(head, H, L, anchor)
    O.verify(toks, np.minimum(target[:1], vocab_rows - 1))
    return case["P"] * vocab_rows / V


def oracle_throughput(case, target, budget_s: float, steps: int | None = None, mode: str = "chain", tree=(0, 0)):
    """Time the oracle on bounded vocabulary slices. Returns (tok/s, sample text, steps run)."""
    V = case["V"]
    # Calibrate the slice so one step costs about budget_s / steps (or ~budget_s/3).
    probe = min(V, 8192)
    t0 = time.perf_counter()
    oracle_cycle_sample(case, probe, target, mode, tree)
    t_probe = time.perf_counter() - t0
    n_steps = steps or 3
    per_step = budget_s / n_steps
    rows = int(min(V, max(1024, probe * per_step / max(t_probe, 1e-6))))
    work = 0.0
    t0 = time.perf_counter()
    done = 0
    for _ in range(n_steps):
        work += oracle_cycle_sample(case, rows, target, mode, tree)
        done += 1
    dt = time.perf_counter() - t0
    what = f"{tree[0]} tree nodes" if mode in ("tree", "marginal") else f"{case['P']} positions"
    sample = (f"1 request, {mode}, {what}, vocabulary rows [0, {rows}) of {V} per step "
              f"(fp64 numpy), {done} steps; units scaled by {rows}/{V}")
    return work / dt, sample, done


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_mode(cfg, variant):
    n_nodes = cfg.get("tree_nodes", 0)
    if n_nodes:
        return ("marginal" if variant == "headoff" else "tree"), (n_nodes, cfg.get("top_m", 0))
    return ("headoff" if variant == "headoff" else "chain"), (0, 0)


# --------------------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from draft_head_gb300 import synth
    cfg = synth.CONFIGS[args.workload]
    case = synth.make_case(cfg, synth.case_seed(args.workload, 0))
    target = synth.make_targets(np.zeros((cfg["batch"], cfg["block"] - 1), np.int64), "uniform", None,
                                cfg["V"], seed=1)
    budget = 150.0
    mode, tree = oracle_mode(cfg, args.variant)
    for _ in range(min(args.warmup, 1)):
        oracle_cycle_sample(case, 1024, target, mode, tree)
    value, sample, done = oracle_throughput(case, target, budget, steps=max(1, args.steps), mode=mode, tree=tree)
    ms = (tree[0] if tree[0] else case["P"]) / value * 1e3
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": done,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(cfg, args.workload, world, args.variant),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores(), "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(cfg, name, world, variant="domino"):
    c = {"workload": name, "d": cfg["d"], "V": cfg["V"], "g": cfg["g"], "e": cfg["e"], "r": cfg["r"],
         "block": cfg["block"], "P": cfg["block"] - 1, "batch_per_gpu": cfg["batch"],
         "global_batch": cfg["batch"] * world, "temperature": cfg["temperature"],
         "parallelism": f"replicas x{world}",
         "l2": "flushed between timed steps (256 MB write, then 256 MB read to retire the dirty lines); W_lm alone (778 MB) exceeds L2"}
    if variant != "domino":
        c["variant"] = variant
    return c




# --------------------------------------------------------------------------- bytes and floors
def step_bytes(cfg, bs, T, sampled, stats=False):
    """Bytes of one chain launch under three countings (per launch, P steps).

    survey: per drafted position every weight the method touches -- W2 (V x r),
        the GRU (W_ih and W_hh, 3g x (e + g)), W1_s (r x g) -- plus each
        request's L_base row and, at T > 0, its noise row;
    substituted: the same with the GRU's input projection taken as one row of
        the prepared gate table (3g fp32 per request) instead of W_ih, b_hh and
        the P_h row added, as the kernels read it (and what the sampled
        verification needs written: the corrected logits, or with stats the
        draft statistics u_i and the row log-partition);
    compulsory: every weight once per launch plus the per-request rows."""
    V, r, g, e, P = cfg["V"], cfg["r"], cfg["g"], cfg["e"], cfg["block"] - 1
    rows = bs * V * 4 * (2 if T > 0 else 1)
    survey = V * r * 2 + 3 * g * (e + g) * 2 + r * g * 2 + rows
    weights = V * r * 2 + 3 * g * g * 2 + r * g * 2 + 3 * g * 2
    out = (bs * (r * 4 + 4) if stats else bs * V * 4) if sampled else 0
    per_req = rows + bs * (r * 4 + 3 * g * 4 + 4) + out
    return {"survey": float(P * survey), "substituted": float(P * (weights + per_req)),
            "compulsory": float(weights + P * per_req)}


def tree_bytes(cfg, bs, N, M, headoff):
    """Bytes of the tree phase (top-M select + best-first build) per launch:
    survey counting -- L_base read once by the select, then per expansion the
    GRU (W_ih and W_hh) and per request the M candidate rows of W2; the
    kernels' own counting reads one gate-table row instead of W_ih."""
    V, r, g, e, P = cfg["V"], cfg["r"], cfg["g"], cfg["e"], cfg["block"] - 1
    top = bs * P * V * 4 + bs * P * M * 8
    nodes = bs * (N + 1) * 16
    if headoff:
        return {"survey": float(top + nodes), "substituted": float(top + nodes), "compulsory": float(top + nodes)}
    per_exp_survey = 3 * g * (e + g) * 2 + r * g * 2 + bs * (M * r * 2)
    per_exp = 3 * g * g * 2 + r * g * 2 + 3 * g * 2 + bs * (3 * g * 4 + r * 4 + M * r * 2)
    return {"survey": float(top + N * per_exp_survey + nodes), "substituted": float(top + N * per_exp + nodes),
            "compulsory": float(top + per_exp + nodes)}


# The multiply-add form of the batch <= 4 chain's W2 GEMV: "ffma2" (packed
# fp32x2 FMAs on unpacked bf16 pairs, one per 64 multiply-adds of a warp) or
# "mma" (bf16 m16n8k16 tensor-core MMAs, one per 16 rows x 16 columns).
SMALL_CHAIN_GEMV = "mma"


def latency_floor(B, cfg, bs, sm_mhz):
    """Lower bound of one small-batch chain step from rates measured on this
    GPU: the W2 GEMV of the busiest SM at the measured issue rate of its
    multiply-add form, plus two one-way trips through L2 (each step's two
    all-to-all exchanges: bottleneck sums, argmax keys)."""
    import torch
    G = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    ws = B.workspace(4096)
    ws.zero_()
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    B.domino_selftest_rates(0, G // 2, out, ws)
    torch.cuda.synchronize()
    cyc, rounds = (int(x) for x in out.cpu())
    one_way = cyc / max(rounds, 1) / 2.0
    rows = -(-cfg["V"] // G)
    iters = 4096
    if SMALL_CHAIN_GEMV == "mma":
        B.domino_selftest_rates(1, iters, out, ws)
        torch.cuda.synchronize()
        per_sm = 16 * iters * 4 / max(int(out[0].item()), 1)  # MMAs per cycle per SM
        gemv = (-(-rows // 16)) * (cfg["r"] // 16) / per_sm
        form = f"bf16 m16n8k16 MMA at {per_sm:.3f} per cycle per SM"
    else:
        B.domino_selftest_rates(2, iters, out, ws)
        torch.cuda.synchronize()
        per_sm = 16 * iters * 16 * 64 / max(int(out[0].item()), 1)  # multiply-adds per cycle per SM
        gemv = rows * cfg["r"] * bs / per_sm
        form = f"packed fp32x2 FMA on bf16 pairs at {per_sm:.1f} multiply-adds per cycle per SM"
    assert B.domino_last_status(ws) == 0
    cycles = gemv + 2.0 * one_way
    return {"us": cycles / sm_mhz, "cycles": cycles, "gemv_cycles": gemv, "exchange_one_way_cycles": one_way,
            "sm_mhz": sm_mhz, "gemv_form": form,
            "rows_per_sm": rows, "note": "GEMV of the busiest SM at the measured issue rate + 2 one-way L2 trips "
                                         "(CTA 0 <-> CTA G/2 flag round trip / 2)"}


# --------------------------------------------------------------------------- one workload
def run_workload(name, args, K, W, rank, world, local, dist, headline, tree_T=0.0):
    """Time one workload: K eager steps (per-phase events), the same step
    replayed K times as one CUDA graph, and for the headline the end-to-end
    cycle from pinned host buffers. Returns the record of this workload."""
    import torch
    from draft_head_gb300 import binding as B
    from draft_head_gb300 import synth
    from draft_head_gb300.runtime import DominoDrafter

    cfg = synth.CONFIGS[name]
    bs, P, V, d, g, r = cfg["batch"], cfg["block"] - 1, cfg["V"], cfg["d"], cfg["g"], cfg["r"]
    T = float(cfg["temperature"])
    case = synth.make_case(cfg, synth.case_seed(name, 0) + 7919 * rank)

    def dev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()

    w = {k: dev(case[k]) for k in ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2")}
    n_nodes, top_m = cfg.get("tree_nodes", 0), cfg.get("top_m", 0)
    is_tree = n_nodes > 0
    drafter = DominoDrafter(w, bs, P, n_nodes, top_m)
    H = dev(case["H"])
    anchor = dev(case["anchor"].astype(np.int32))
    headoff = args.variant == "headoff"
    sampled = T > 0 and not is_tree and not headoff  # T > 0: standard speculative sampling verification
    # The sampled verification works from the chain's draft statistics (no
    # [batch, P, V] draft logits) from batch 5 on, where the batched chain
    # runs anyway; below, the small-batch chain and its logits are faster.
    stats = sampled and bs >= 5 and drafter.stats_supported()
    target = torch.zeros(bs, P, dtype=torch.int32, device="cuda")
    if sampled:
        Zt = dev(synth.normal((bs, P + 1, V), 1.0, 4242, 0))  # the target's logits (synthetic)
        Ut = dev(synth.uniform_open01((bs, P), 4242, 1).astype(np.float32))
        Gt = dev(synth.gumbel_noise((bs, V), 4243))
    if is_tree:
        tnext = torch.zeros(bs, n_nodes + 1, dtype=torch.int32, device="cuda")
    gumbel = dev(case["gumbel"]) if T > 0 else None
    gview = gumbel[:, 1:, :] if gumbel is not None else None
    gstride = cfg["block"] * V if gumbel is not None else 0
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device="cuda")

    def l2_flush():
        # Write 256 MB (evicts every line), then read another 256 MB so the
        # dirty lines of the write are written back here, outside the timed
        # region, and not during the next step's first kernel.
        flush_w.zero_()
        flush_r.sum()

    def head_pass():
        # The sequential part of the step: the chain (or the best-first tree).
        if is_tree:
            drafter.tree_marginal(anchor, tree_T) if headoff else drafter.tree(anchor, tree_T)
        elif headoff:
            drafter.chain_headoff(T, gview, gstride)
        else:
            if stats:
                drafter.chain_stats(anchor, T, gview, gstride)
            else:
                drafter.chain(anchor, T, gview, gstride, logits_out=drafter.draft_logits() if sampled else None)

    def tail_pass():
        # Acceptance: the longest matching prefix of the block, or the tree walk.
        if is_tree:
            drafter.tree_verify(tnext, want_path=True, want_mask=True)
        elif stats:
            drafter.verify_sampled_head(Zt, Ut, Gt, T)
        elif sampled:
            drafter.verify_sampled(Zt, Ut, Gt, T)
        else:
            drafter.verify(target)

    def step():
        drafter.base(H)
        head_pass()
        tail_pass()

    # The workload's targets follow its draft: flip / match each drafted token
    # with the configured probability (the tree: the first-popped child's
    # token w.p. 0.8); drawn once from the first draft, then fixed.
    drafter.base(H)
    head_pass()
    torch.cuda.synchronize()
    mode, p_t = cfg.get("target", ("uniform", None))
    if is_tree:
        tnext_np = synth.make_tree_targets(drafter.node_token.cpu().numpy(), drafter.node_parent.cpu().numpy(),
                                           0.2, V, seed=4)
        tnext.copy_(torch.from_numpy(tnext_np))
        target_np = np.zeros((bs, P), np.int32)
    else:
        target_np = synth.make_targets(drafter.tokens.cpu().numpy(), mode, p_t, V, seed=3)
        target.copy_(torch.from_numpy(target_np))
        target_desc = f"{mode} {p_t}" if p_t is not None else mode

    for _ in range(W):
        l2_flush()
        step()
    torch.cuda.synchronize()
    assert drafter.last_status() == 0, "device-side error during warm-up"

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for k in range(K):
        l2_flush()  # outside the timed events
        e = ev[k]
        e[0].record()
        drafter.base(H)
        e[1].record()
        head_pass()
        e[2].record()
        tail_pass()
        e[3].record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    assert drafter.last_status() == 0, "device-side error in the timed region"

    t_base = [e[0].elapsed_time(e[1]) for e in ev]
    t_chain = [e[1].elapsed_time(e[2]) for e in ev]
    t_ver = [e[2].elapsed_time(e[3]) for e in ev]
    t_step = [e[0].elapsed_time(e[3]) for e in ev]
    total_ms = max_over_ranks(float(sum(t_step)), dist, "cuda")
    per_step = bs * (n_nodes if is_tree else P)  # drafted tokens (tree: drafted nodes) per step
    value = replica_throughput(per_step * K, world, total_ms)

    # Acceptance of the last timed step (same inputs every step).
    if is_tree:
        acc = drafter.accept.cpu().numpy().astype(int)
        accept = {"per_request": acc.tolist(), "mean_accept": float(acc.mean()),
                  "mean_tokens_advanced": float(acc.mean() + 1.0),
                  "targets": "first-popped child's token w.p. 0.8 per node, else a token none of its children's"}
    else:
        acc = drafter.accept.cpu().numpy().astype(int)
        accept = {"per_request": acc.tolist(), "mean_accept": float(acc.mean()),
                  "mean_tokens_advanced": float(acc.mean() + 1.0),
                  "targets": ("standard speculative sampling against synthetic target logits N(0, 1)"
                              if sampled else f"{target_desc} of the draft, per position iid")}

    peaks = measured_peaks()
    base_bytes = float(V * d * 2 + r * d * 2 + bs * P * d * 2 + bs * P * V * 4 + bs * P * r * 4)
    base_flops = 2.0 * bs * P * (V + r) * d
    if is_tree:
        hb = tree_bytes(cfg, bs, n_nodes, top_m, headoff)
    elif headoff:
        x = float(bs * P * V * 4 * (2 if T > 0 else 1) + bs * P * 4)
        hb = {"survey": x, "substituted": x, "compulsory": x}
    else:
        hb = step_bytes(cfg, bs, T, sampled, stats)
    avg_base = statistics.mean(t_base) * 1e-3
    avg_chain = statistics.mean(t_chain) * 1e-3
    avg_ver = statistics.mean(t_ver) * 1e-3
    hbm = peaks["hbm_gbs"] * 1e9
    head_name = "dominotree" if is_tree else "draft_chain"
    phases = {
        "base_logits": {"ms": avg_base * 1e3, "bytes": base_bytes, "flops": base_flops,
                        "gbs": base_bytes / avg_base / 1e9, "hbm_frac": base_bytes / avg_base / hbm,
                        "tflops": base_flops / avg_base / 1e12,
                        "tc_frac": base_flops / avg_base / 1e12 / peaks["bf16_tflops"]},
        head_name: {"ms": avg_chain * 1e3, "bytes_survey": hb["survey"], "bytes_substituted": hb["substituted"],
                    "bytes_compulsory": hb["compulsory"],
                    "hbm_frac_survey": hb["survey"] / avg_chain / hbm,
                    "hbm_frac_substituted": hb["substituted"] / avg_chain / hbm,
                    "hbm_frac_compulsory": hb["compulsory"] / avg_chain / hbm},
        "verify": {"ms": avg_ver * 1e3},
    }
    if not is_tree:
        phases[head_name]["step_us"] = avg_chain / P * 1e6
    dominant = "base_logits" if avg_base >= avg_chain else head_name
    if dominant == "base_logits":
        tc_bound = base_flops / (peaks["bf16_tflops"] * 1e12) > base_bytes / hbm
        kname = "gemm_bf16_tc (base logits)"
        if tc_bound:
            roof = {"kernel": kname, "bound": "tensor", "achieved": base_flops / avg_base / 1e12,
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
        else:
            roof = {"kernel": kname, "bound": "hbm", "achieved": base_bytes / avg_base / 1e9,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        tr = recorded_traffic("gemm_bf16_tc", name)
        roof["traffic"] = tr
        roof["algorithmic_bytes_per_launch"] = base_bytes
        if tr:
            roof["frac_dram"] = tr / avg_base / hbm
    else:
        kname = ("headoff_chain_kernel" if not is_tree else "topm + tree_marginal_kernel") if headoff else \
            ("topm + tree_kernel" if is_tree else chain_kernel_name(cfg, bs))
        tr = recorded_traffic(kname, name)
        roof = {"kernel": kname, "bound": "hbm", "achieved": hb["survey"] / avg_chain / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "traffic": tr,
                "algorithmic_bytes_per_launch": hb["survey"],
                "frac_substituted": hb["substituted"] / avg_chain / hbm,
                "frac_compulsory": hb["compulsory"] / avg_chain / hbm,
                "frac_dram": (tr / avg_chain / hbm) if tr else None}
        if kname == "chain_small_kernel":
            roof["note"] = ("achieved counts the survey's per-step bytes (W2, W_ih + W_hh, W1_s and the request "
                            "rows at every step); this kernel keeps W2 and W_hh on chip for the whole chain and "
                            "reads a gate-table row instead of W_ih, so its DRAM traffic is near the compulsory "
                            "bytes and the HBM rate does not bound it: two dependent all-to-all exchanges per "
                            "step do (latency_floor_us)")
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = peaks["source"]

    # ---------------- the same step, captured once as a CUDA graph and replayed
    # K times (the headline): the same kernels on the same inputs, the L2
    # flush between replays outside the events; the launch gaps of the eager
    # loop above are what it removes. Phases and the roofline come from the
    # eager loop's per-kernel events.
    graph, graph_note = None, None
    t_wall2 = t_wall1
    if not args.no_graph:
        try:
            gr = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                step()
            torch.cuda.current_stream().wait_stream(side)
            with torch.cuda.graph(gr):
                step()
            for _ in range(max(3, W)):
                l2_flush()
                gr.replay()
            torch.cuda.synchronize()
            gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
            if dist:
                dist.barrier()
            torch.cuda.synchronize()
            for k in range(K):
                l2_flush()
                gev[k][0].record()
                gr.replay()
                gev[k][1].record()
            torch.cuda.synchronize()
            t_wall2 = time.time()
            if dist:
                dist.barrier()
            assert drafter.last_status() == 0, "device-side error in the graph replays"
            g_ms = max_over_ranks(float(sum(a.elapsed_time(b) for a, b in gev)), dist, "cuda")
            graph = {"value": replica_throughput(per_step * K, world, g_ms), "ms_per_step": g_ms / K}
        except (RuntimeError, AssertionError) as ex:
            graph_note = f"graph capture failed ({type(ex).__name__}); eager launches reported"
            torch.cuda.synchronize()
    clocks = sampler.stop(t_wall0, t_wall2) if sampler else None

    floor = None
    if not is_tree and not headoff and kname == "chain_small_kernel":
        mhz = (clocks or {}).get("sm_mhz") or 2070.0
        floor = latency_floor(B, cfg, bs, mhz)
        roof["latency_floor_us"] = floor["us"]
        roof["latency_frac"] = floor["us"] / (avg_chain / P * 1e6)

    # Kernels of this library per step: base GEMM; chain: scratch reset + chain
    # (head-off: one argmax kernel); tree: scratch reset + three top-M passes +
    # the build (marginal tree: no reset); then the acceptance kernel (one, at
    # T > 0 too).
    if is_tree:
        launches_per_step = 1 + (3 + 1 if headoff else 1 + 3 + 1) + 1
    elif headoff:
        launches_per_step = 1 + 1 + 1
    else:
        launches_per_step = 1 + 2 + 1

    eager = {"value": value, "ms_per_step": total_ms / K}
    if graph:
        timing = ("each step replayed as one captured CUDA graph (base pass, chain or tree, acceptance); "
                  "phases and roofline from the same steps launched eagerly (see 'eager')")
        value, step_ms = graph["value"], graph["ms_per_step"]
    else:
        timing = graph_note or "eager launches"
        step_ms = total_ms / K
    rec = {"value": value, "unit": UNIT, "ms_per_step": step_ms, "steps": K, "warmup": W,
           "dtype": "bf16" if cfg["dtype"] == "bf16" else "f32",
           "config": workload_config(cfg, name, world, args.variant),
           "phases": phases, "roofline": roof, "accept": accept, "clocks": clocks, "timing": timing,
           "eager": eager, "launches_per_step": launches_per_step}
    if is_tree:
        rec["config"]["tree_scoring_temperature"] = tree_T
        rec["config"]["tree"] = {"nodes": n_nodes, "top_m": top_m}
    else:
        rec["chain_step_latency_us"] = avg_chain / P * 1e6
        if floor:
            rec["latency_floor_us"] = floor
    if not headline:
        del drafter, w, H
        torch.cuda.empty_cache()
        return rec

    # ---------------- end to end through the public API: pinned host in, host out.
    e2e = None
    e2e_note = "eager"
    if not args.no_e2e:
        Hh = torch.from_numpy(case["H"].view(np.int16) if case["H"].dtype == np.uint16 else case["H"]).pin_memory()
        if case["H"].dtype == np.uint16:
            Hh = Hh.view(torch.bfloat16)
        ah = torch.from_numpy(case["anchor"].astype(np.int32)).pin_memory()
        th = torch.from_numpy(target_np).pin_memory()
        tok_h = torch.empty(bs, P, dtype=torch.int32).pin_memory()
        acc_h = torch.empty(bs, dtype=torch.int32).pin_memory()
        Hd, ad, td = torch.empty_like(H), torch.empty_like(anchor), torch.empty_like(target)
        Ke = min(K, 200)
        if is_tree:
            tok_h = torch.empty(bs, n_nodes + 1, dtype=torch.int32).pin_memory()
            par_h = torch.empty(bs, n_nodes + 1, dtype=torch.int32).pin_memory()
            tnh = torch.from_numpy(tnext_np).pin_memory()
            tnd = torch.empty_like(tnext)

        def host_cycle():
            if is_tree:
                Hd.copy_(Hh, non_blocking=True)
                ad.copy_(ah, non_blocking=True)
                tnd.copy_(tnh, non_blocking=True)
                drafter.base(Hd)
                drafter.tree_marginal(ad, tree_T) if headoff else drafter.tree(ad, tree_T)
                drafter.tree_verify(tnd, want_path=True, want_mask=False)
                tok_h.copy_(drafter.node_token, non_blocking=True)
                par_h.copy_(drafter.node_parent, non_blocking=True)
                acc_h.copy_(drafter.accept, non_blocking=True)
            elif headoff:
                Hd.copy_(Hh, non_blocking=True)
                td.copy_(th, non_blocking=True)
                drafter.base(Hd)
                drafter.chain_headoff(T, gview, gstride)
                drafter.verify(td)
                tok_h.copy_(drafter.tokens, non_blocking=True)
                acc_h.copy_(drafter.accept, non_blocking=True)
            elif sampled:
                # The target's logits are produced on the device by the target pass.
                Hd.copy_(Hh, non_blocking=True)
                ad.copy_(ah, non_blocking=True)
                drafter.base(Hd)
                if stats:
                    drafter.chain_stats(ad, T, gview, gstride)
                    drafter.verify_sampled_head(Zt, Ut, Gt, T)
                else:
                    drafter.chain(ad, T, gview, gstride, logits_out=drafter.draft_logits())
                    drafter.verify_sampled(Zt, Ut, Gt, T)
                tok_h.copy_(drafter.tokens, non_blocking=True)
                acc_h.copy_(drafter.accept, non_blocking=True)
            elif host_graph:
                drafter.replay_io_cycle()
            else:
                drafter.cycle_io(io, T, gview, gstride)

        # The chain cycle moves its inputs and results through packed pinned
        # buffers (one copy each way) and goes through the captured cycle
        # (copies and kernels as one CUDA graph) when capture works here.
        host_graph = False
        io = None
        if not (is_tree or headoff or sampled):
            from draft_head_gb300.runtime import HostIO
            io = HostIO(drafter, d, H.dtype)
            io.H_host.copy_(Hh)
            io.anchor_host.copy_(ah)
            io.target_host.copy_(th)
            try:
                drafter.capture_io_cycle(io, T, gview, gstride)
                host_graph = True
            except Exception as ex:  # reported in the JSON line
                e2e_note = f"eager (graph capture failed: {type(ex).__name__})"
        for _ in range(3):
            host_cycle()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        host_s = 0.0
        cur = torch.cuda.current_stream()
        for k in range(Ke):
            l2_flush()
            cur.synchronize()  # the flush is done before the host clock starts
            h0 = time.perf_counter()
            evs[k][0].record()
            host_cycle()
            evs[k][1].record()
            cur.synchronize()  # tokens and accept lengths readable on the host
            host_s += time.perf_counter() - h0
        e_ms = max_over_ranks(float(sum(a.elapsed_time(b) for a, b in evs)), dist, "cuda")
        h_ms = max_over_ranks(host_s * 1e3, dist, "cuda")
        if is_tree:
            h2d = Hh.numel() * Hh.element_size() + ah.numel() * 4 + tnh.numel() * 4
            d2h = tok_h.numel() * 4 + par_h.numel() * 4 + acc_h.numel() * 4
        elif headoff:
            h2d = Hh.numel() * Hh.element_size() + th.numel() * 4
            d2h = tok_h.numel() * 4 + acc_h.numel() * 4
        elif sampled:
            h2d = Hh.numel() * Hh.element_size() + ah.numel() * 4
            d2h = tok_h.numel() * 4 + acc_h.numel() * 4
        else:  # the packed buffers, alignment padding included
            h2d = io.host_in.numel()
            d2h = io.host_out.numel() * 4
        e2e = {"value": replica_throughput(per_step * Ke, world, e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": Ke,
               "host_wall": {"value": replica_throughput(per_step * Ke, world, h_ms), "ms_per_step": h_ms / Ke,
                             "what": "host clock from the launch of the cycle (inputs ready in pinned memory) "
                                     "to its results readable on the host after a stream synchronize"},
               "mode": "one CUDA graph: one packed host-to-device copy, kernels, one device-to-host copy" if host_graph
               else e2e_note}
    rec["e2e"] = e2e
    rec["_case"] = (case, target_np)
    return rec


# --------------------------------------------------------------------------- main arm
EXTRA_WORKLOADS = [("qwen3_4b_bs64", 0.0), ("qwen3_8b_bs32", 0.0), ("qwen3_4b_tree", 0.0), ("qwen3_4b_tree", 0.5)]


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from draft_head_gb300 import synth

    K, W = args.steps, args.warmup
    head = run_workload(args.workload, args, K, W, rank, world, local, dist, headline=True,
                        tree_T=args.tree_temperature)
    case, target_np = head.pop("_case")
    cfg = synth.CONFIGS[args.workload]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        mode, tree = oracle_mode(cfg, args.variant)
        v, sample, _ = oracle_throughput(case, target_np, 15.0, mode=mode, tree=tree)
        cpu = {"value": v, "unit": UNIT, "cores": cores(), "cpu_model": cpu_model(), "kind": "oracle",
               "sample": sample}
    del case

    # The other workloads of the method, at one GPU only (the scaling runs keep
    # the headline alone): fewer steps each, same warm-up and L2 flush rules.
    workloads = {}
    if world == 1 and not args.no_workloads:
        Kw, Ww = max(10, min(K, 60)), max(3, min(W, 5))
        for name, tT in EXTRA_WORKLOADS:
            if name == args.workload and tT == args.tree_temperature:
                continue
            key = name if not synth.CONFIGS[name].get("tree_nodes") else f"{name}_T{tT:g}"
            try:
                rec = run_workload(name, args, Kw, Ww, rank, world, local, dist, headline=False, tree_T=tT)
                rec.pop("_case", None)
                workloads[key] = rec
            except (RuntimeError, AssertionError) as ex:
                workloads[key] = {"error": f"{type(ex).__name__}: {ex}"}
            torch.cuda.empty_cache()

    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": W, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
                "data": "synthetic", "config": head["config"],
                "chain_step_latency_us": head.get("chain_step_latency_us"),
                "latency_floor_us": head.get("latency_floor_us"),
                "phases": head["phases"], "roofline": head["roofline"], "accept": head["accept"],
                "cpu_baseline": cpu, "e2e": head["e2e"], "gpu_launches": head["launches_per_step"] * K,
                "clocks": head["clocks"], "timing": head["timing"], "eager": head["eager"],
                "workloads": workloads}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
