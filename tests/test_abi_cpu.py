"""C-ABI checks that need no GPU: the library loads, exports every function
include/domino.h declares, and rejects bad arguments on the host before
anything is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from draft_head_gb300 import build
    build.build()
    from draft_head_gb300 import binding
    return binding


def declared_functions():
    src = open(os.path.join(ROOT, "include", "domino.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:domino|dominotree)_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(B):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(B.lib, n), n
    assert set(names) == set(B.EXPORTED)


def test_abi_version_and_status_strings(B):
    assert B.domino_abi_version() == 3
    for code, name in B.STATUS.items():
        assert B.domino_status_str(code) == name
    assert B.domino_status_str(99) == "DOMINO_ERR_UNKNOWN"


def _fake_head(B, dtype=1, d=2560, e=2560, g=1024, r=256, V=151936, table=True):
    fake = 0x100000  # never dereferenced: validation rejects before any launch
    h = B.domino_head(dtype, d, e, g, r, V, *([fake] * 8), fake if table else None)
    return h


def test_host_validation(B):
    lib = B.lib
    h = _fake_head(B)
    ref = ctypes.byref(h)
    null = None
    # null head
    assert lib.domino_base_logits(None, 0x100000, 1, 15, 0x100000, None, 0x100000, 4096, null) == 1
    # bad dtype
    hb = _fake_head(B, dtype=7)
    assert lib.domino_base_logits(ctypes.byref(hb), 0x100000, 1, 15, 0x100000, None, 0x100000, 4096, null) == 1
    # rank above the kernels' limit
    hr = _fake_head(B, r=512)
    assert lib.domino_base_logits(ctypes.byref(hr), 0x100000, 1, 15, 0x100000, None, 0x100000, 4096, null) == 2
    # bf16 dims must be multiples of 8
    hd = _fake_head(B, d=2561)
    assert lib.domino_base_logits(ctypes.byref(hd), 0x100000, 1, 15, 0x100000, None, 0x100000, 4096, null) == 2
    # misaligned weight pointer
    hm = _fake_head(B)
    hm.w2 = 0x100004
    assert lib.domino_base_logits(ctypes.byref(hm), 0x100000, 1, 15, 0x100000, None, 0x100000, 4096, null) == 1
    # chain without a prepared gate table
    hn = _fake_head(B, table=False)
    assert lib.domino_draft_chain(ctypes.byref(hn), 0x100000, 0x100000, 0x100000, 1, 15, 0.0, None, 0, None,
                                  0x100000, None, 0x100000, 1 << 30, null) == 1
    # chain: sampling needs noise; negative temperature rejected; workspace too small / misaligned
    assert lib.domino_draft_chain(ref, 0x100000, 0x100000, 0x100000, 1, 15, 1.0, None, 0, None,
                                  0x100000, None, 0x100000, 1 << 30, null) == 1
    assert lib.domino_draft_chain(ref, 0x100000, 0x100000, 0x100000, 1, 15, -1.0, None, 0, None,
                                  0x100000, None, 0x100000, 1 << 30, null) == 1
    assert lib.domino_draft_chain(ref, 0x100000, 0x100000, 0x100000, 1, 15, 0.0, None, 0, None,
                                  0x100000, None, 0x100000, 16, null) == 5
    assert lib.domino_draft_chain(ref, 0x100000, 0x100000, 0x100000, 1, 15, 0.0, None, 0, None,
                                  0x100000, None, 0x100010, 1 << 30, null) == 5
    # empty batch is a no-op
    assert lib.domino_draft_chain(ref, None, None, None, 0, 15, 0.0, None, 0, None, None, None, None, 0,
                                  null) == 0
    assert lib.domino_verify(None, None, 0, 15, None, None, null) == 0
    assert lib.domino_verify(None, None, -1, 15, None, None, null) == 1
    # top-M limits
    assert lib.domino_topm_select(0x100000, 2, 100, 0, 0x100000, None, 0x100000, 1 << 20, null) == 1
    assert lib.domino_topm_select(0x100000, 2, 100, 257, 0x100000, None, 0x100000, 1 << 20, null) == 1
    assert lib.domino_topm_select(0x100000, 2, 100, 101, 0x100000, None, 0x100000, 1 << 20, null) == 1
    # tree limits
    assert lib.dominotree_build(ref, 0x100000, 0x100000, 0x100000, 16, 15, 0, 64, 0.0, 0x100000, 0x100000,
                                0x100000, 0x100000, 0x100000, 1 << 30, null) == 1
    assert lib.dominotree_build(ref, 0x100000, 0x100000, 0x100000, 16, 15, 65, 64, 0.0, 0x100000, 0x100000,
                                0x100000, 0x100000, 0x100000, 1 << 30, null) == 1
    assert lib.dominotree_build(ref, 0x100000, 0x100000, 0x100000, 16, 15, 16, 64, 0.0, 0x100000, 0x100000,
                                0x100000, 0x100000, None, 0, null) == 5
    # the scoring temperature: >= 0 and finite
    for bad_t in (-0.5, float("nan"), float("inf")):
        assert lib.dominotree_build(ref, 0x100000, 0x100000, 0x100000, 16, 15, 16, 64, bad_t, 0x100000,
                                    0x100000, 0x100000, 0x100000, 0x100000, 1 << 30, null) == 1
        assert lib.dominotree_build_marginal(0x100000, 0x100000, 16, 15, 1000, 16, 64, bad_t, 0x100000,
                                             0x100000, 0x100000, 0x100000, 0x100000, 1 << 30, null) == 1
    # last_status needs an aligned workspace
    assert lib.domino_last_status(None, null) == 5
    # chain statistics: both outputs required, u 16-byte aligned; empty batch is a no-op
    F = 0x100000
    assert lib.domino_draft_chain_stats(ref, F, F, F, 8, 15, 1.0, F, 15 * 151936, None, F, None, F, F, 1 << 30,
                                        null) == 1
    assert lib.domino_draft_chain_stats(ref, F, F, F, 8, 15, 1.0, F, 15 * 151936, None, F, F + 4, F, F, 1 << 30,
                                        null) == 1
    assert lib.domino_draft_chain_stats(ref, None, None, None, 0, 15, 1.0, None, 0, None, None, None, None, None, 0,
                                        null) == 0
    # an fp32 head has no batched chain: no statistics
    hf = _fake_head(B, dtype=0)
    assert lib.domino_draft_chain_stats_supported(ctypes.byref(hf), 8, 15) == 0
    assert lib.domino_draft_chain_stats_supported(ref, 0, 15) == 0
    # head-form verification: T > 0, the statistics present, a bf16 rank-256 head
    ws_h = lib.domino_verify_sampled_head_workspace_bytes(8, 15)
    assert ws_h >= 256 + 8 * 4 + 8 * 8 + 8 * 8 and ws_h % 256 == 0
    for bad_t in (0.0, -1.0, float("nan")):
        assert lib.domino_verify_sampled_head(ref, F, F, F, F, F, F, F, 8, 15, bad_t, F, F, F, F, ws_h, null) == 1
    assert lib.domino_verify_sampled_head(ref, F, F, None, F, F, F, F, 8, 15, 1.0, F, F, F, F, ws_h, null) == 1
    assert lib.domino_verify_sampled_head(ref, F, F, F + 8, F, F, F, F, 8, 15, 1.0, F, F, F, F, ws_h, null) == 1
    assert lib.domino_verify_sampled_head(ctypes.byref(hf), F, F, F, F, F, F, F, 8, 15, 1.0, F, F, F, F, ws_h,
                                          null) == 2
    h128 = _fake_head(B, r=128)
    assert lib.domino_verify_sampled_head(ctypes.byref(h128), F, F, F, F, F, F, F, 8, 15, 1.0, F, F, F, F, ws_h,
                                          null) == 2
    assert lib.domino_verify_sampled_head(ref, F, F, F, F, F, F, F, 8, 15, 1.0, F, F, F, F, ws_h - 256, null) == 5
    assert lib.domino_verify_sampled_head(ref, None, None, None, None, None, None, None, 0, 15, 1.0, None, None,
                                          None, None, 0, null) == 0


def test_workspace_sizes(B):
    h = _fake_head(B)
    a = B.lib.domino_workspace_bytes(ctypes.byref(h), 1, 15, 0, 0)
    b = B.lib.domino_workspace_bytes(ctypes.byref(h), 64, 15, 0, 0)
    c = B.lib.domino_workspace_bytes(ctypes.byref(h), 16, 15, 16, 64)
    assert 256 < a < b and c > a
    assert a % 256 == 0 and b % 256 == 0
    # per row: a threshold key, a count (padded block), a 4096-key candidate list
    al = lambda x: (x + 255) // 256 * 256
    assert B.lib.domino_topm_workspace_bytes(240, 151936, 64) == al(240 * 8 + al(240 * 4) + 240 * 4096 * 8)


def test_checked_build_exports_the_same_symbols():
    """libdomino_checked.so (device-side index checks, -DDOMINO_CHECKED) loads
    without a GPU and exports exactly what the header declares."""
    import ctypes
    import os
    from draft_head_gb300 import build as bld
    from draft_head_gb300 import binding as B
    path = bld.build(checked=True)
    lib = ctypes.CDLL(path)
    for name in B.EXPORTED:
        assert hasattr(lib, name), name
    lib.domino_status_str.restype = ctypes.c_char_p
    assert lib.domino_status_str(7) == b"DOMINO_ERR_INDEX"
    assert os.path.basename(path) == "libdomino_checked.so"
