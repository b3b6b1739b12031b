"""Thin ctypes binding of libdomino (include/domino.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels. The functions carry the C names; tensors are torch tensors on
the current CUDA device and are passed by data pointer, streams default to
torch's current stream. A non-OK status raises DominoError. If the compiled
library is missing this module raises at import time -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# DOMINO_LIB=checked loads the checked build (device-side index checks that
# report DOMINO_ERR_INDEX instead of touching memory out of range).
LIB_NAME = "libdomino_checked.so" if os.environ.get("DOMINO_LIB", "") == "checked" else "libdomino.so"
LIB_PATH = os.path.join(_PKG, "lib", LIB_NAME)

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_NAME} not built ({LIB_PATH}); run `python -m draft_head_gb300.build`")

lib = ctypes.CDLL(LIB_PATH)

F32, BF16 = 0, 1
STATUS = {0: "DOMINO_OK", 1: "DOMINO_ERR_INVALID_ARG", 2: "DOMINO_ERR_UNSUPPORTED", 3: "DOMINO_ERR_CUDA",
          4: "DOMINO_ERR_TIMEOUT", 5: "DOMINO_ERR_WORKSPACE", 6: "DOMINO_ERR_DEVICE_DATA", 7: "DOMINO_ERR_INDEX"}

EXPORTED = [
    "domino_abi_version", "domino_status_str", "domino_workspace_bytes", "domino_prepare_gate_table",
    "domino_base_logits", "domino_draft_chain", "domino_verify", "domino_topm_workspace_bytes",
    "domino_topm_select", "dominotree_build", "domino_last_status", "domino_set_wait_timeout_ns",
    "domino_selftest_wait_timeout", "domino_draft_chain_noalloc", "dominotree_verify", "domino_selftest_rates",
    "domino_headoff_workspace_bytes", "domino_draft_chain_headoff", "dominotree_build_marginal",
    "domino_verify_sampled_workspace_bytes", "domino_verify_sampled",
    "domino_draft_chain_stats_supported", "domino_draft_chain_stats",
    "domino_verify_sampled_head_workspace_bytes", "domino_verify_sampled_head",
]


class DominoError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class domino_head(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("d", ctypes.c_int32), ("e", ctypes.c_int32),
                ("g", ctypes.c_int32), ("r", ctypes.c_int32), ("V", ctypes.c_int32),
                ("w_lm", ctypes.c_void_p), ("emb", ctypes.c_void_p), ("w_ih", ctypes.c_void_p),
                ("w_hh", ctypes.c_void_p), ("b_ih", ctypes.c_void_p), ("b_hh", ctypes.c_void_p),
                ("w1", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("gate_table", ctypes.c_void_p)]


_vp, _i32, _i64, _sz, _f32, _u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                    ctypes.c_float, ctypes.c_uint64)
_HP = ctypes.POINTER(domino_head)


def _sig(name, res, args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = args
    return f


_sig("domino_abi_version", _i32, [])
_sig("domino_status_str", ctypes.c_char_p, [_i32])
_sig("domino_workspace_bytes", _sz, [_HP, _i32, _i32, _i32, _i32])
_sig("domino_prepare_gate_table", _i32, [_HP, _vp, _vp, _sz, _vp])
_sig("domino_base_logits", _i32, [_HP, _vp, _i32, _i32, _vp, _vp, _vp, _sz, _vp])
_sig("domino_draft_chain", _i32, [_HP, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _i64, _vp, _vp, _vp, _vp,
                                  _sz, _vp])
_sig("domino_verify", _i32, [_vp, _vp, _i32, _i32, _vp, _vp, _vp])
_sig("domino_topm_workspace_bytes", _sz, [_i32, _i32, _i32])
_sig("domino_topm_select", _i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp])
_sig("dominotree_build", _i32, [_HP, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _vp, _vp,
                                _sz, _vp])
_sig("domino_last_status", _i32, [_vp, _vp])
_sig("domino_set_wait_timeout_ns", None, [_u64])
_sig("domino_selftest_wait_timeout", _i32, [_u64, _vp, _sz, _vp])
_sig("domino_selftest_rates", _i32, [_i32, _i32, _vp, _vp, _sz, _vp])
_sig("domino_draft_chain_noalloc", _i32, [_HP, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _i64, _vp, _vp, _vp, _vp,
                                          _vp])
_sig("domino_verify_sampled_workspace_bytes", _sz, [_i32, _i32])
_sig("domino_verify_sampled", _i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _vp, _sz,
                                     _vp])
_sig("domino_draft_chain_stats_supported", _i32, [_HP, _i32, _i32])
_sig("domino_draft_chain_stats", _i32, [_HP, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _i64, _vp, _vp, _vp, _vp, _vp,
                                        _sz, _vp])
_sig("domino_verify_sampled_head_workspace_bytes", _sz, [_i32, _i32])
_sig("domino_verify_sampled_head", _i32, [_HP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp,
                                          _vp, _sz, _vp])
_sig("dominotree_verify", _i32, [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp])
_sig("domino_headoff_workspace_bytes", _sz, [_i32, _i32, _i32, _i32, _i32])
_sig("domino_draft_chain_headoff", _i32, [_vp, _i32, _i32, _i32, _f32, _vp, _i64, _vp, _vp, _sz, _vp])
_sig("dominotree_build_marginal", _i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _vp, _vp, _vp,
                                         _sz, _vp])


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st, where):
    if st != 0:
        raise DominoError(st, where)


class Head:
    """Owns a domino_head struct built from device tensors (kept alive here).

    Weights: uint16/bfloat16 tensors for bf16 heads, float32 for f32 heads."""

    def __init__(self, w_lm, emb, w_ih, w_hh, b_ih, b_hh, w1, w2, gate_table=None):
        dt = BF16 if w_lm.dtype in (torch.bfloat16, torch.int16, torch.uint16) else F32
        V, d = w_lm.shape
        e = emb.shape[1]
        g = w_hh.shape[1]
        r = w1.shape[0]
        self.tensors = dict(w_lm=w_lm, emb=emb, w_ih=w_ih, w_hh=w_hh, b_ih=b_ih, b_hh=b_hh, w1=w1, w2=w2)
        self.gate_table = gate_table
        self.c = domino_head(dt, d, e, g, r, V, *[_ptr(self.tensors[k]) for k in
                                                  ("w_lm", "emb", "w_ih", "w_hh", "b_ih", "b_hh", "w1", "w2")],
                             _ptr(gate_table))
        self.dtype, self.d, self.e, self.g, self.r, self.V = dt, d, e, g, r, V

    def set_gate_table(self, table):
        self.gate_table = table
        self.c.gate_table = _ptr(table)

    def ref(self):
        return ctypes.byref(self.c)


def domino_abi_version() -> int:
    return lib.domino_abi_version()


def domino_status_str(status: int) -> str:
    return lib.domino_status_str(status).decode()


def domino_workspace_bytes(head: Head, batch: int, P: int, n_nodes: int = 0, top_m: int = 0) -> int:
    return lib.domino_workspace_bytes(head.ref(), batch, P, n_nodes, top_m)


def domino_prepare_gate_table(head: Head, table, ws, stream=None):
    _check(lib.domino_prepare_gate_table(head.ref(), _ptr(table), _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(stream)), "domino_prepare_gate_table")


def domino_base_logits(head: Head, H, batch: int, P: int, L_base, P_h, ws, stream=None):
    _check(lib.domino_base_logits(head.ref(), _ptr(H), batch, P, _ptr(L_base), _ptr(P_h), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)), "domino_base_logits")


def domino_draft_chain(head: Head, L_base, P_h, anchor, batch: int, P: int, temperature: float, gumbel,
                       gumbel_batch_stride: int, force_tokens, tokens, logits_out, ws, stream=None):
    _check(lib.domino_draft_chain(head.ref(), _ptr(L_base), _ptr(P_h), _ptr(anchor), batch, P,
                                  float(temperature), _ptr(gumbel), int(gumbel_batch_stride),
                                  _ptr(force_tokens), _ptr(tokens), _ptr(logits_out), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)), "domino_draft_chain")


def domino_draft_chain_stats_supported(head: Head, batch: int, P: int) -> bool:
    return bool(lib.domino_draft_chain_stats_supported(head.ref(), batch, P))


def domino_draft_chain_stats(head: Head, L_base, P_h, anchor, batch: int, P: int, temperature: float, gumbel,
                             gumbel_batch_stride: int, force_tokens, tokens, u_out, lse_out, ws, stream=None):
    _check(lib.domino_draft_chain_stats(head.ref(), _ptr(L_base), _ptr(P_h), _ptr(anchor), batch, P,
                                        float(temperature), _ptr(gumbel), int(gumbel_batch_stride),
                                        _ptr(force_tokens), _ptr(tokens), _ptr(u_out), _ptr(lse_out), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)), "domino_draft_chain_stats")


def domino_verify(draft, target, batch: int, P: int, accept_len, advanced, stream=None):
    _check(lib.domino_verify(_ptr(draft), _ptr(target), batch, P, _ptr(accept_len), _ptr(advanced),
                             _stream(stream)), "domino_verify")


def domino_topm_workspace_bytes(rows: int, n: int, top_m: int) -> int:
    return lib.domino_topm_workspace_bytes(rows, n, top_m)


def domino_topm_select(values, rows: int, n: int, top_m: int, ids_out, vals_out, ws, stream=None):
    _check(lib.domino_topm_select(_ptr(values), rows, n, top_m, _ptr(ids_out), _ptr(vals_out), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)), "domino_topm_select")


def dominotree_build(head: Head, L_base, P_h, anchor, batch: int, P: int, n_nodes: int, top_m: int,
                     node_token, node_parent, node_depth, node_score, ws, stream=None, temperature: float = 0.0):
    _check(lib.dominotree_build(head.ref(), _ptr(L_base), _ptr(P_h), _ptr(anchor), batch, P, n_nodes, top_m,
                                float(temperature), _ptr(node_token), _ptr(node_parent), _ptr(node_depth), _ptr(node_score),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "dominotree_build")


def domino_last_status(ws, stream=None) -> int:
    return lib.domino_last_status(_ptr(ws), _stream(stream))


def domino_set_wait_timeout_ns(ns: int):
    lib.domino_set_wait_timeout_ns(int(ns))


def domino_selftest_wait_timeout(timeout_ns: int, ws, stream=None):
    _check(lib.domino_selftest_wait_timeout(int(timeout_ns), _ptr(ws), ws.numel() * ws.element_size(),
                                            _stream(stream)), "domino_selftest_wait_timeout")


def domino_selftest_rates(which: int, arg: int, out, ws, stream=None):
    """Diagnostic rates behind the chain's latency floor (see domino.h);
    out: device int64 [2]."""
    _check(lib.domino_selftest_rates(int(which), int(arg), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)), "domino_selftest_rates")


def workspace(nbytes: int, device=None):
    """A zeroed device workspace tensor (torch's allocator returns 256-byte
    aligned blocks; the status word must start at zero)."""
    n = max(256, (int(nbytes) + 255) // 256 * 256)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def domino_draft_chain_noalloc(head: Head, L_base, P_h, anchor, batch: int, P: int, temperature: float, gumbel,
                               gumbel_batch_stride: int, force_tokens, tokens, logits_out, device_status=None,
                               stream=None):
    """domino_draft_chain with the library's fixed scratch (no workspace argument)."""
    _check(lib.domino_draft_chain_noalloc(head.ref(), _ptr(L_base), _ptr(P_h), _ptr(anchor), batch, P,
                                          float(temperature), _ptr(gumbel), int(gumbel_batch_stride),
                                          _ptr(force_tokens), _ptr(tokens), _ptr(logits_out),
                                          _ptr(device_status), _stream(stream)), "domino_draft_chain_noalloc")


def dominotree_verify(node_token, node_parent, target_next, batch: int, n_nodes: int, accept_len, advanced,
                      accepted_path=None, mask=None, stream=None):
    _check(lib.dominotree_verify(_ptr(node_token), _ptr(node_parent), _ptr(target_next), batch, n_nodes,
                                 _ptr(accept_len), _ptr(advanced), _ptr(accepted_path), _ptr(mask),
                                 _stream(stream)), "dominotree_verify")


def domino_headoff_workspace_bytes(batch: int, P: int, V: int, n_nodes: int = 0, top_m: int = 0) -> int:
    return lib.domino_headoff_workspace_bytes(batch, P, V, n_nodes, top_m)


def domino_draft_chain_headoff(L_base, batch: int, P: int, V: int, temperature: float, gumbel,
                               gumbel_batch_stride: int, tokens, ws, stream=None):
    _check(lib.domino_draft_chain_headoff(_ptr(L_base), batch, P, V, float(temperature), _ptr(gumbel),
                                          int(gumbel_batch_stride), _ptr(tokens), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream)),
           "domino_draft_chain_headoff")


def dominotree_build_marginal(L_base, anchor, batch: int, P: int, V: int, n_nodes: int, top_m: int, node_token,
                              node_parent, node_depth, node_score, ws, stream=None, temperature: float = 0.0):
    _check(lib.dominotree_build_marginal(_ptr(L_base), _ptr(anchor), batch, P, V, n_nodes, top_m,
                                         float(temperature), _ptr(node_token), _ptr(node_parent), _ptr(node_depth),
                                         _ptr(node_score), _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(stream)), "dominotree_build_marginal")


def domino_verify_sampled_workspace_bytes(batch: int, P: int) -> int:
    return lib.domino_verify_sampled_workspace_bytes(batch, P)


def domino_verify_sampled(draft, draft_logits, target_logits, uniform, gumbel, batch: int, P: int, V: int,
                          temperature: float, accept_len, advanced, next_token, ws, stream=None):
    _check(lib.domino_verify_sampled(_ptr(draft), _ptr(draft_logits), _ptr(target_logits), _ptr(uniform),
                                     _ptr(gumbel), batch, P, V, float(temperature), _ptr(accept_len),
                                     _ptr(advanced), _ptr(next_token), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)), "domino_verify_sampled")


def domino_verify_sampled_head_workspace_bytes(batch: int, P: int) -> int:
    return lib.domino_verify_sampled_head_workspace_bytes(batch, P)


def domino_verify_sampled_head(head: Head, draft, L_base, u, lse, target_logits, uniform, gumbel, batch: int, P: int,
                               temperature: float, accept_len, advanced, next_token, ws, stream=None):
    _check(lib.domino_verify_sampled_head(head.ref(), _ptr(draft), _ptr(L_base), _ptr(u), _ptr(lse),
                                          _ptr(target_logits), _ptr(uniform), _ptr(gumbel), batch, P,
                                          float(temperature), _ptr(accept_len), _ptr(advanced), _ptr(next_token),
                                          _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "domino_verify_sampled_head")
