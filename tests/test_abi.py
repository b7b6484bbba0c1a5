"""The C-ABI library loads, exports every symbol the header declares, and rejects bad arguments on the host
before anything is launched (no GPU needed: validation runs before the first CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dominotree.h")

OK, INVALID, UNSUPPORTED = 0, 1, 2
A = 1 << 20  # a 16-byte-aligned fake device address: validation must reject before any dereference


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(dt_[a-z_0-9]+)\s*\(", text))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert {"dt_topm", "dt_build_trees", "dt_topm_workspace_bytes", "dt_build_workspace_bytes", "dt_get_error",
            "dt_workspace_init", "dt_status_string"} <= names


def test_library_exports_every_declared_symbol(dtlib):
    L = dtlib.lib()
    names = declared_functions()
    assert names == set(dtlib.SIGNATURES), "binding signatures and header declarations diverge"
    for name in names:
        assert getattr(L, name) is not None
    nm = subprocess.run(["nm", "-D", "--defined-only", str(dtlib.buildlib.LIB)], capture_output=True, text=True)
    exported = set(re.findall(r"\b(dt_[a-z_0-9]+)\b", nm.stdout))
    assert names <= exported
    assert L.dt_abi_version() == 1


def test_status_strings(dtlib):
    L = dtlib.lib()
    for s in range(6):
        assert L.dt_status_string(s)
    assert L.dt_status_string(99) == b"unknown status"


def test_workspace_sizes(dtlib):
    t = dtlib.dt_topm_workspace_bytes
    assert t(1, 4, 1024, 8) >= 256 and t(1, 4, 1024, 8) % 256 == 0
    # per (row, chunk of 16384 logits): a candidate count and room for max(64, 4M) 8-byte candidate words
    assert t(1, 16, 151936, 64) >= 256 + 16 * 10 * (4 + 256 * 8)   # 10 chunks of 16384 logits per row
    assert t(256, 16, 151936, 128) > t(64, 16, 151936, 64)
    b = dtlib.dt_build_workspace_bytes
    assert b(32, 16, 151936, 64, 32, 1024, 4096) >= 32 * 32 * 1024 * 4 + t(32, 16, 151936, 64)
    # the round's workspace holds the top-M region first, then the builder's own region
    assert b(2, 4, 20000, 8, 16, 64, 64) > t(2, 4, 20000, 8)
    assert t(-1, 1, 1, 1) == 0 and b(1, 1, 1, 1, 0, 8, 8) == 0


def _topm(L, logits=A, dtype=1, B=1, K=2, V=100, M=5, ids=A, vals=A, ws=A, wsb=1 << 30):
    return L.dt_topm(logits, dtype, B, K, V, M, ids, vals, ws, wsb, None)


def test_topm_rejects_bad_arguments(dtlib):
    L = dtlib.lib()
    assert _topm(L, M=0) == INVALID
    assert _topm(L, M=101) == INVALID
    assert _topm(L, K=0) == INVALID
    assert _topm(L, B=-1) == INVALID
    assert _topm(L, dtype=7) == INVALID
    assert _topm(L, logits=None) == INVALID
    assert _topm(L, logits=A + 8) == INVALID          # misaligned
    assert _topm(L, ws=A + 4) == INVALID
    assert _topm(L, wsb=16) == INVALID                # workspace too small
    assert _topm(L, V=5000, M=2000) == UNSUPPORTED    # M above DT_MAX_M
    assert _topm(L, B=0) == OK                        # nothing to do, nothing launched


def test_static_topm_rejects_bad_arguments(dtlib):
    """dt_topm_static's own checks, all made on the host before any CUDA call (no GPU here)."""
    L = dtlib.lib()

    def call(logits=A, dtype=1, B=1, K=2, V=100, M=5, ids=A, vals=A):
        return L.dt_topm_static(logits, dtype, B, K, V, M, ids, vals, None)
    assert call(M=0) == INVALID
    assert call(M=101) == INVALID                     # more candidates than vocabulary
    assert call(K=0) == INVALID
    assert call(B=-1) == INVALID
    assert call(dtype=7) == INVALID
    assert call(logits=None) == INVALID
    assert call(ids=None) == INVALID
    assert call(vals=None) == INVALID
    assert call(logits=A + 8) == INVALID              # misaligned
    assert call(ids=A + 4) == INVALID
    assert call(vals=A + 2) == INVALID
    assert call(V=5000, M=2000) == UNSUPPORTED        # M above DT_MAX_M
    # beyond the fixed array: the limits are per dtype (fp32 words are twice as wide and its chunks half as long)
    assert call(dtype=0, B=1, K=818, V=151936, M=64) == UNSUPPORTED
    assert call(dtype=1, B=1, K=3247, V=151936, M=64) == UNSUPPORTED
    assert call(dtype=1, B=1, K=1631, V=151936, M=128) == UNSUPPORTED
    assert call(B=0) == OK                            # nothing to do, nothing launched


def _weights(dtlib, H=32, E=32, dtype=1, b_ih=None, emb=A):
    return dtlib._Weights(H, E, dtype, emb, A, A, b_ih, None, A)


def _build(dtlib, B=1, K=4, V=100, M=4, n=8, max_depth=3, T=0.0, w=None, ws=A, wsb=1 << 30):
    w = w or _weights(dtlib)
    return dtlib.lib().dt_build_trees(B, K, V, M, n, max_depth, T, A, A, A, ctypes.byref(w), A, A, A, A, A, ws, wsb,
                                      None)


def test_build_rejects_bad_arguments(dtlib):
    assert _build(dtlib, max_depth=5) == INVALID                 # deeper than the block
    assert _build(dtlib, M=2, max_depth=2, n=7) == INVALID       # 2 + 4 = 6 nodes exist
    assert _build(dtlib, M=2, max_depth=2, n=6, B=0) == OK       # exactly the whole tree is allowed
    assert _build(dtlib, T=-0.5) == INVALID
    assert _build(dtlib, T=float("nan")) == INVALID
    assert _build(dtlib, T=float("inf")) == INVALID
    assert _build(dtlib, w=_weights(dtlib, H=30)) == INVALID     # H not a multiple of 8
    assert _build(dtlib, w=_weights(dtlib, E=12)) == INVALID
    assert _build(dtlib, w=_weights(dtlib, dtype=3)) == INVALID
    assert _build(dtlib, w=_weights(dtlib, emb=None)) == INVALID
    assert _build(dtlib, w=_weights(dtlib, b_ih=A + 2)) == INVALID
    assert _build(dtlib, M=0) == INVALID
    assert _build(dtlib, M=200, V=100) == INVALID
    assert _build(dtlib, n=0) == INVALID
    assert _build(dtlib, wsb=64) == INVALID
    assert _build(dtlib, w=_weights(dtlib, H=4096)) == UNSUPPORTED
    assert _build(dtlib, M=2000, V=5000) == UNSUPPORTED
    assert dtlib.lib().dt_build_trees(1, 4, 100, 4, 8, 3, 0.0, A, A, A, None, A, A, A, A, A, A, 1 << 30,
                                      None) == INVALID
    assert _build(dtlib, B=0) == OK


def test_round_rejects_bad_arguments(dtlib):
    L = dtlib.lib()

    def rnd(B=1, K=4, V=100, M=4, n=8, max_depth=3, T=0.0, w=None, dtype=1, logits=A, wsb=1 << 30):
        w = w or _weights(dtlib)
        return L.dt_round(logits, dtype, B, K, V, M, n, max_depth, T, A, ctypes.byref(w), A, A, A, A, A, A, A, A, wsb,
                          None)

    assert rnd(logits=None) == INVALID                      # the top-M's checks
    assert rnd(dtype=7) == INVALID
    assert rnd(M=2000, V=5000) == UNSUPPORTED
    assert rnd(max_depth=5) == INVALID                      # the builder's
    assert rnd(T=-1.0) == INVALID
    assert rnd(w=_weights(dtlib, H=30)) == INVALID
    assert rnd(wsb=64) == INVALID
    assert rnd(B=0) == OK                                   # nothing to do, nothing launched


def test_binding_refuses_host_tensors(dtlib):
    import torch
    with pytest.raises(TypeError):
        dtlib.dt_topm(torch.zeros(1, 2, 64), 4, out_ids=torch.zeros(1, 2, 4, dtype=torch.int32),
                      out_vals=torch.zeros(1, 2, 4), workspace=torch.zeros(4096, dtype=torch.uint8))


def test_build_stats_reject_bad_arguments(dtlib):
    L = dtlib.lib()
    st = dtlib._BuildStats()
    assert L.dt_build_stats_read(None, ctypes.byref(st), None) == INVALID
    assert L.dt_build_stats_read(A + 8, ctypes.byref(st), None) == INVALID   # misaligned
    assert L.dt_build_stats_read(A, None, None) == INVALID


def test_lookahead_setting_is_validated(dtlib):
    L = dtlib.lib()
    assert L.dt_set_lookahead(-1) == INVALID
    assert L.dt_set_lookahead(9) == INVALID
    for k in (1, 8, 0):
        assert L.dt_set_lookahead(k) == OK


def test_topm_cluster_setting_is_validated(dtlib):
    L = dtlib.lib()
    assert L.dt_set_topm_cluster(-1) == INVALID
    assert L.dt_set_topm_cluster(2) == INVALID
    for v in (0, 1):
        assert L.dt_set_topm_cluster(v) == OK


def test_marginal_rejects_bad_arguments(dtlib):
    L = dtlib.lib()
    f = L.dt_build_trees_marginal
    good = dict(B=1, K=4, V=100, M=5, n=8, max_depth=4, T=0.0)

    def call(**kw):
        a = dict(good, **kw)
        return f(a["B"], a["K"], a["V"], a["M"], a["n"], a["max_depth"], a["T"], A, A, A, A, A, A, A, A,
                 kw.get("wsb", 1 << 20), None)
    assert call(M=0) == INVALID
    assert call(M=101) == INVALID
    assert call(max_depth=5) == INVALID
    assert call(T=-1.0) == INVALID
    assert call(n=10 ** 6, M=2, max_depth=2) == INVALID     # more nodes than the depth-limited tree has
    assert call(wsb=16) == INVALID                           # no room for the status word
    assert call(M=2000, V=5000) == UNSUPPORTED
    assert f(1, 4, 100, 5, 8, 4, 0.0, A, A, A, A, A, A, A + 8, A, 1 << 20, None) == INVALID  # misaligned
    assert call(B=0) == OK


def test_accept_rejects_bad_arguments(dtlib):
    f = dtlib.lib().dt_accept_paths
    assert f(1, 0, A, A, A, A, A, A, None) == INVALID
    assert f(-1, 4, A, A, A, A, A, A, None) == INVALID
    assert f(1, 4, A + 2, A, A, A, A, A, None) == INVALID
    assert f(1, 4, None, A, A, A, A, A, None) == INVALID
    assert f(1, 2000, A, A, A, A, A, A, None) == UNSUPPORTED
    assert f(0, 4, A, A, A, A, A, A, None) == OK


def test_lmhead_rejects_bad_arguments(dtlib):
    f = dtlib.lib().dt_lmhead_topm
    BF16, F32 = 1, 0

    def call(R=16, D=128, V=1000, M=8, dtype=BF16, h=A, w=A, ids=A, vals=A, ws=A):
        return f(R, D, V, M, h, w, dtype, ids, vals, ws, 1 << 30, None)
    assert call(M=0) == INVALID
    assert call(M=1001) == INVALID                    # more candidates than vocabulary
    assert call(R=-1) == INVALID
    assert call(D=0) == INVALID
    assert call(dtype=7) == INVALID
    assert call(h=None) == INVALID
    assert call(w=A + 8) == INVALID                   # misaligned
    assert call(dtype=F32) == UNSUPPORTED             # the tensor-core path takes bf16
    assert call(D=96) == UNSUPPORTED                  # K blocks of 64
    assert call(R=8193) == UNSUPPORTED                # every row's bound and count in shared memory
    assert call(M=2000, V=5000) == UNSUPPORTED
    assert call(R=0) == OK


def test_tree_attention_rejects_bad_arguments(dtlib):
    f = dtlib.lib().dt_tree_attention
    BF16, F32 = 1, 0

    def call(B=1, n=16, L=100, Hq=32, Hkv=8, d=128, dtype=BF16, q=A, mask=A, scale=0.088, ws=A):
        return f(B, n, L, Hq, Hkv, d, q, A, A, dtype, mask, scale, A, ws, 1 << 30, None)
    assert call(Hq=30) == INVALID                     # not a multiple of the key/value heads
    assert call(n=0) == INVALID
    assert call(L=-1) == INVALID
    assert call(scale=0.0) == INVALID
    assert call(scale=float("nan")) == INVALID
    assert call(q=None) == INVALID
    assert call(q=A + 4) == INVALID                   # misaligned
    assert call(mask=None) == INVALID
    assert call(dtype=7) == INVALID
    assert call(dtype=F32) == UNSUPPORTED             # the tensor-core path takes bf16
    assert call(d=64) == UNSUPPORTED
    assert call(n=17) == UNSUPPORTED                  # 4 query heads per key/value head x 17 nodes > 64 rows
    assert call(B=0) == OK


def test_packed_buffers_align_every_view(dtlib):
    """The host-round buffers: every view starts on a 16-byte boundary (the C ABI's rule) and they do not overlap."""
    import torch
    buf, v = dtlib.packed_buffers([("a", (3, 5), torch.int32), ("b", (7,), torch.uint8), ("c", (2, 3), torch.float32),
                                   ("d", (1, 16, 16), torch.uint8)], "cpu")
    base = buf.data_ptr()
    spans = []
    for name, t in v.items():
        off = t.data_ptr() - base
        assert off % 16 == 0, name
        spans.append((off, off + t.numel() * t.element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    assert spans[-1][1] <= buf.numel()
    v["c"][1, 2] = 1.5
    assert v["c"][1, 2].item() == 1.5 and v["a"].shape == (3, 5) and v["d"].dtype == torch.uint8


def test_workspace_calls_reject_bad_arguments(dtlib):
    """The workspace's own calls check their pointer and size on the host, before any CUDA call."""
    L = dtlib.lib()
    assert L.dt_workspace_init(None, 1 << 20, None) == INVALID
    assert L.dt_workspace_init(A + 8, 1 << 20, None) == INVALID   # misaligned
    assert L.dt_workspace_init(A, 16, None) == INVALID            # smaller than the status header
    assert L.dt_get_error(None, None) == INVALID
    assert L.dt_get_error(A + 4, None) == INVALID


def test_device_sized_workspaces_reject_empty_shapes(dtlib):
    """The projection's and the tree attention's workspace sizes depend on the device (its SM count); shapes with
    nothing to compute get 0 before the device is asked."""
    L = dtlib.lib()
    for args in [(0, 64, 1000, 8), (16, 0, 1000, 8), (16, 64, 0, 8), (16, 64, 1000, 0)]:
        assert L.dt_lmhead_workspace_bytes(*args) == 0, args
    for args in [(0, 16, 128, 32, 8, 128), (1, 0, 128, 32, 8, 128), (1, 16, -1, 32, 8, 128), (1, 16, 128, 0, 8, 128),
                 (1, 16, 128, 32, 0, 128), (1, 16, 128, 32, 8, 0)]:
        assert L.dt_tree_attention_workspace_bytes(*args) == 0, args
