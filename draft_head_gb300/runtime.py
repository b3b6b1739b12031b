"""DominoDrafter: owns the device buffers of one drafting configuration and
drives the C-ABI entry points for a speculative cycle (base pass, chain,
verification). Buffer management and argument marshalling only; every
computation runs in libdomino's kernels.
"""
from __future__ import annotations

import torch

from . import binding as B


class DominoDrafter:
    def __init__(self, weights: dict, batch: int, P: int, n_nodes: int = 0, top_m: int = 0,
                 device="cuda"):
        """weights: device tensors w_lm, emb, w_ih, w_hh, b_ih, b_hh, w1, w2
        (bf16 or fp32). Prepares the GRU gate table once."""
        self.dev = torch.device(device)
        self.head = B.Head(weights["w_lm"], weights["emb"], weights["w_ih"], weights["w_hh"],
                           weights["b_ih"], weights["b_hh"], weights["w1"], weights["w2"])
        h = self.head
        self.batch, self.P, self.n_nodes, self.top_m = batch, P, n_nodes, top_m
        self.ws = B.workspace(B.domino_workspace_bytes(h, batch, P, n_nodes, top_m), self.dev)
        self.gate_table = torch.empty(h.V * 3 * h.g, dtype=torch.float32, device=self.dev)
        B.domino_prepare_gate_table(h, self.gate_table, self.ws)
        h.set_gate_table(self.gate_table)
        self.L_base = torch.empty(batch, P, h.V, dtype=torch.float32, device=self.dev)
        self.P_h = torch.empty(batch, P, h.r, dtype=torch.float32, device=self.dev)
        # Drafted tokens and accept lengths share one device buffer (the accept
        # lengths 16-byte aligned after the tokens), so a cycle's results
        # leave in one device-to-host copy.
        self._acc_off = (batch * P + 3) // 4 * 4
        self._out = torch.empty(self._acc_off + batch, dtype=torch.int32, device=self.dev)
        self.tokens = self._out[: batch * P].view(batch, P)
        self.accept = self._out[self._acc_off: self._acc_off + batch]
        self.advanced = torch.empty(batch, dtype=torch.int32, device=self.dev)
        if n_nodes > 0:
            shape = (batch, n_nodes + 1)
            self.node_token = torch.empty(shape, dtype=torch.int32, device=self.dev)
            self.node_parent = torch.empty(shape, dtype=torch.int32, device=self.dev)
            self.node_depth = torch.empty(shape, dtype=torch.int32, device=self.dev)
            self.node_score = torch.empty(shape, dtype=torch.float32, device=self.dev)

    def base(self, H):
        B.domino_base_logits(self.head, H, self.batch, self.P, self.L_base, self.P_h, self.ws)

    def chain(self, anchor, temperature=0.0, gumbel=None, gumbel_batch_stride=0, force=None,
              logits_out=None):
        B.domino_draft_chain(self.head, self.L_base, self.P_h, anchor, self.batch, self.P, temperature,
                             gumbel, gumbel_batch_stride, force, self.tokens, logits_out, self.ws)
        return self.tokens

    def draft(self, H, anchor, temperature=0.0, gumbel=None, gumbel_batch_stride=0):
        self.base(H)
        return self.chain(anchor, temperature, gumbel, gumbel_batch_stride)

    def tree(self, anchor, temperature=0.0):
        """DominoTree best-first build over the current base pass; children
        scored by log-softmax(l / T) over the slice (T = 1 at temperature 0)."""
        B.dominotree_build(self.head, self.L_base, self.P_h, anchor, self.batch, self.P, self.n_nodes,
                           self.top_m, self.node_token, self.node_parent, self.node_depth, self.node_score,
                           self.ws, temperature=temperature)
        return self.node_token, self.node_parent, self.node_depth, self.node_score

    def draft_logits(self):
        """Device buffer [batch, P, V] fp32 for the chain's corrected logits
        (pass it as chain(..., logits_out=...) before verify_sampled)."""
        if not hasattr(self, "logits"):
            self.logits = torch.empty(self.batch, self.P, self.head.V, dtype=torch.float32, device=self.dev)
        return self.logits

    def verify_sampled(self, target_logits, uniform, gumbel_next, temperature):
        """Verification at T > 0 of the current draft against the target's
        logits [batch, P + 1, V] (domino_verify_sampled): returns accept,
        advanced and the next token drawn from the target side."""
        if not hasattr(self, "ws_sampled"):
            self.ws_sampled = B.workspace(B.domino_verify_sampled_workspace_bytes(self.batch, self.P), self.dev)
        if not hasattr(self, "next_token"):
            self.next_token = torch.empty(self.batch, dtype=torch.int32, device=self.dev)
        B.domino_verify_sampled(self.tokens, self.draft_logits(), target_logits, uniform, gumbel_next, self.batch,
                                self.P, self.head.V, temperature, self.accept, self.advanced, self.next_token,
                                self.ws_sampled)
        return self.accept, self.advanced, self.next_token

    def stats_supported(self):
        """True when the chain can return its draft statistics (u_i and the
        row log-partitions) in place of the logits: the batched tensor-core
        chain's shapes (at batch <= 4 the logits form is the faster one)."""
        return B.domino_draft_chain_stats_supported(self.head, self.batch, self.P)

    def chain_stats(self, anchor, temperature, gumbel=None, gumbel_batch_stride=0, force=None):
        """The chain with the draft statistics instead of the logits
        (domino_draft_chain_stats): tokens, u [batch, P, r], lse [batch, P]."""
        if not hasattr(self, "u_stats"):
            self.u_stats = torch.empty(self.batch, self.P, self.head.r, dtype=torch.float32, device=self.dev)
            self.lse_stats = torch.empty(self.batch, self.P, dtype=torch.float32, device=self.dev)
        B.domino_draft_chain_stats(self.head, self.L_base, self.P_h, anchor, self.batch, self.P, temperature, gumbel,
                                   gumbel_batch_stride, force, self.tokens, self.u_stats, self.lse_stats, self.ws)
        return self.tokens, self.u_stats, self.lse_stats

    def verify_sampled_head(self, target_logits, uniform, gumbel_next, temperature):
        """Verification at T > 0 from the head and the chain's statistics
        (domino_verify_sampled_head; run chain_stats first): accept, advanced,
        next token."""
        if not hasattr(self, "ws_sampled_head"):
            self.ws_sampled_head = B.workspace(B.domino_verify_sampled_head_workspace_bytes(self.batch, self.P),
                                               self.dev)
        if not hasattr(self, "next_token"):
            self.next_token = torch.empty(self.batch, dtype=torch.int32, device=self.dev)
        B.domino_verify_sampled_head(self.head, self.tokens, self.L_base, self.u_stats, self.lse_stats, target_logits,
                                     uniform, gumbel_next, self.batch, self.P, temperature, self.accept,
                                     self.advanced, self.next_token, self.ws_sampled_head)
        return self.accept, self.advanced, self.next_token

    def tree_verify(self, target_next, want_path=True, want_mask=False):
        """Tree acceptance of the current tree (dominotree_verify): target_next
        [batch, n_nodes + 1] int32, the target's greedy next token per node."""
        N1 = self.n_nodes + 1
        if want_path and not hasattr(self, "tree_path"):
            self.tree_path = torch.empty(self.batch, N1, dtype=torch.int32, device=self.dev)
        if want_mask and not hasattr(self, "tree_mask"):
            self.tree_mask = torch.empty(self.batch, N1, N1, dtype=torch.uint8, device=self.dev)
        path = self.tree_path if want_path else None
        mask = self.tree_mask if want_mask else None
        B.dominotree_verify(self.node_token, self.node_parent, target_next, self.batch, self.n_nodes,
                            self.accept, self.advanced, path, mask)
        return self.accept, self.advanced, path, mask

    def _headoff_ws(self):
        if not hasattr(self, "ws_headoff"):
            self.ws_headoff = B.workspace(B.domino_headoff_workspace_bytes(
                self.batch, self.P, self.head.V, self.n_nodes, self.top_m), self.dev)
        return self.ws_headoff

    def chain_headoff(self, temperature=0.0, gumbel=None, gumbel_batch_stride=0):
        """The head-off baseline: per-position argmax of the base logits."""
        B.domino_draft_chain_headoff(self.L_base, self.batch, self.P, self.head.V, temperature, gumbel,
                                     gumbel_batch_stride, self.tokens, self._headoff_ws())
        return self.tokens

    def tree_marginal(self, anchor, temperature=0.0):
        """The marginal-scored best-first tree over the current base pass."""
        B.dominotree_build_marginal(self.L_base, anchor, self.batch, self.P, self.head.V, self.n_nodes,
                                    self.top_m, self.node_token, self.node_parent, self.node_depth,
                                    self.node_score, self._headoff_ws(), temperature=temperature)
        return self.node_token, self.node_parent, self.node_depth, self.node_score

    def verify(self, target):
        B.domino_verify(self.tokens, target, self.batch, self.P, self.accept, self.advanced)
        return self.accept, self.advanced

    def cycle_from_host(self, H_host, anchor_host, target_host, out_tokens_host, out_accept_host,
                        H_dev, anchor_dev, target_dev, temperature=0.0, gumbel=None, gumbel_batch_stride=0):
        """One cycle from pinned host inputs to pinned host results, all stream-ordered."""
        H_dev.copy_(H_host, non_blocking=True)
        anchor_dev.copy_(anchor_host, non_blocking=True)
        target_dev.copy_(target_host, non_blocking=True)
        self.draft(H_dev, anchor_dev, temperature, gumbel, gumbel_batch_stride)
        self.verify(target_dev)
        out_tokens_host.copy_(self.tokens, non_blocking=True)
        out_accept_host.copy_(self.accept, non_blocking=True)

    def capture_host_cycle(self, H_host, anchor_host, target_host, out_tokens_host, out_accept_host,
                           H_dev, anchor_dev, target_dev, temperature=0.0, gumbel=None, gumbel_batch_stride=0):
        """Capture cycle_from_host (pinned host inputs in, pinned host results
        out: three copies, the kernels, two copies) as one CUDA graph;
        replay_host_cycle() reruns it with whatever the pinned buffers hold
        at replay time. The cycle runs once, uncaptured, first."""
        args = (H_host, anchor_host, target_host, out_tokens_host, out_accept_host, H_dev, anchor_dev, target_dev,
                temperature, gumbel, gumbel_batch_stride)
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):
            self.cycle_from_host(*args)
        torch.cuda.current_stream(self.dev).wait_stream(side)
        self.host_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.host_graph):
            self.cycle_from_host(*args)
        return self.host_graph

    def replay_host_cycle(self):
        """Rerun the captured host cycle on the current stream."""
        self.host_graph.replay()

    def cycle_io(self, io: "HostIO", temperature=0.0, gumbel=None, gumbel_batch_stride=0):
        """One cycle through packed pinned buffers (HostIO): the inputs go to
        the device in one copy, the drafted tokens and accept lengths come
        back in one; all stream-ordered."""
        io.dev_in.copy_(io.host_in, non_blocking=True)
        self.draft(io.H, io.anchor, temperature, gumbel, gumbel_batch_stride)
        self.verify(io.target)
        io.host_out.copy_(self._out, non_blocking=True)

    def capture_io_cycle(self, io: "HostIO", temperature=0.0, gumbel=None, gumbel_batch_stride=0):
        """Capture cycle_io as one CUDA graph (two copies and the kernels);
        replay_io_cycle() reruns it with whatever io.host_in holds at replay
        time. The cycle runs once, uncaptured, first."""
        args = (io, temperature, gumbel, gumbel_batch_stride)
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):
            self.cycle_io(*args)
        torch.cuda.current_stream(self.dev).wait_stream(side)
        self.io_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.io_graph):
            self.cycle_io(*args)
        return self.io_graph

    def replay_io_cycle(self):
        """Rerun the captured packed-buffer cycle on the current stream."""
        self.io_graph.replay()


    def capture_cycle(self, H, anchor, target, temperature=0.0, gumbel=None, gumbel_batch_stride=0):
        """Capture one drafting cycle (base pass, chain, verify) on these device
        tensors into a CUDA graph; replay() reruns it, reading whatever the
        tensors hold at replay time. The cycle runs once, uncaptured, first."""
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):
            self.draft(H, anchor, temperature, gumbel, gumbel_batch_stride)
            self.verify(target)
        torch.cuda.current_stream(self.dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.draft(H, anchor, temperature, gumbel, gumbel_batch_stride)
            self.verify(target)
        return self.graph

    def replay(self):
        """Rerun the captured cycle on the current stream."""
        self.graph.replay()
        return self.tokens, self.accept

    def last_status(self) -> int:
        return B.domino_last_status(self.ws)


class HostIO:
    """Pinned host buffers for one drafting cycle of a DominoDrafter, packed
    so that the cycle moves its inputs to the device in one copy and its
    results back in one. host_in holds H [batch, P, d] (dtype of the head's
    activations), the anchor [batch] int32 and the target tokens [batch, P]
    int32, each section 16-byte aligned; H_host, anchor_host and target_host
    are views into it, and H, anchor, target the matching device views.
    host_out mirrors the drafter's result buffer: tokens_host [batch, P] and
    accept_host [batch]."""

    def __init__(self, drafter: DominoDrafter, d: int, h_dtype=torch.bfloat16):
        bs, P = drafter.batch, drafter.P
        al = lambda x: (x + 15) // 16 * 16
        esz = torch.empty(0, dtype=h_dtype).element_size()
        n_h = bs * P * d * esz
        o_a = al(n_h)
        o_t = al(o_a + bs * 4)
        total = al(o_t + bs * P * 4)
        self.host_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.dev_in = torch.empty(total, dtype=torch.uint8, device=drafter.dev)

        def views(buf):
            return (buf[:n_h].view(h_dtype).view(bs, P, d), buf[o_a:o_a + bs * 4].view(torch.int32),
                    buf[o_t:o_t + bs * P * 4].view(torch.int32).view(bs, P))

        self.H_host, self.anchor_host, self.target_host = views(self.host_in)
        self.H, self.anchor, self.target = views(self.dev_in)
        self.host_out = torch.empty(drafter._out.numel(), dtype=torch.int32).pin_memory()
        self.tokens_host = self.host_out[: bs * P].view(bs, P)
        self.accept_host = self.host_out[drafter._acc_off: drafter._acc_off + bs]
