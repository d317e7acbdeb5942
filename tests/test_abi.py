"""The C-ABI library loads and exports every entry point include/txl.h declares;
host-side validation rejects bad arguments before anything reaches a GPU.
CPU only: no call here launches a kernel."""

import ctypes
import os
import re

import pytest
import torch

import transformer_xl_relative_pos_gb300 as txl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "txl.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, SHAPE, CUDA, TIMEOUT, WORKSPACE = 0, -1, -2, -3, -4, -5, -6, -7


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(txl_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("txl_rel_pos_emb", "txl_relattn_fwd", "txl_mem_update", "txl_mem_concat",
              "txl_status_string", "txl_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(txl.lib_path() if os.path.exists(txl.lib_path()) else txl.build.build())
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in txl.h but not exported"


def test_status_strings_and_version():
    assert txl.status_string(OK) == "ok"
    assert "timed out" in txl.status_string(TIMEOUT)
    assert txl.status_string(12345) == "unknown status"
    assert txl.version() >= 100


def test_workspace_size_arithmetic():
    assert txl.workspace_size(16, 16, 128, 64, 1) == 0
    rows = 16 * 16 * 128
    o = 3 * rows * 64 * 4
    o = (o + 255) // 256 * 256
    assert txl.workspace_size(16, 16, 128, 64, 3) == o + 3 * rows * 4


def test_relattn_plan_validation_and_routing():
    # Host arithmetic only.  Without a GPU the SM count is taken as GB300's 152.
    k, n = ctypes.c_int(0), ctypes.c_int(0)
    plan = txl.lib().txl_relattn_plan
    assert plan(1, 16, 100, 4, 104, 64, txl.BF16, 0, 0, None, ctypes.byref(n)) == INVALID
    assert plan(1, 16, 100, 4, 103, 64, txl.BF16, 0, 0, ctypes.byref(k), ctypes.byref(n)) == SHAPE
    assert plan(1, 16, 100, 4, 104, 32, txl.BF16, 0, 0, ctypes.byref(k), ctypes.byref(n)) == UNSUPPORTED
    assert plan(1, 16, 100, 0, 100, 64, txl.BF16, 0, 0, ctypes.byref(k), ctypes.byref(n)) == INVALID
    assert plan(1, 16, 100, 4, 104, 64, 7, 0, 0, ctypes.byref(k), ctypes.byref(n)) == INVALID
    assert plan(1, 1, 16, 16, 32, 64, txl.F32, 2, 0, ctypes.byref(k), ctypes.byref(n)) == UNSUPPORTED
    assert txl.relattn_plan(1, 1, 16, 16, torch.float32) == ("f32", 1)
    ws = 1 << 30
    # Segments past eight queries take the tensor cores; the headline shape
    # (256 query tiles on 152 SMs) is not split.
    assert txl.relattn_plan(16, 16, 1600, 128, workspace_bytes=ws) == ("tc", 1)
    assert txl.relattn_plan(8, 16, 3800, 9, workspace_bytes=ws)[0] == "tc"
    assert txl.relattn_plan(1, 16, 3800, 9, workspace_bytes=0)[0] == "tc"
    # Up to eight queries always a decode kernel, whatever the batch, memory
    # or workspace (one query on the CUDA cores, more on warp MMAs); an explicit
    # split counts its key ranges.
    assert txl.relattn_plan(8, 16, 3800, 6, n_splits=3, workspace_bytes=ws) == ("decode_mma", 3)
    assert txl.relattn_plan(8, 16, 3800, 1, n_splits=3, workspace_bytes=ws) == ("decode", 3)
    for B, M, L in [(8, 3800, 1), (2, 800, 6), (1, 3800, 6), (1, 12000, 8), (64, 3800, 8), (1, 5, 2)]:
        want = "decode" if L == 1 else "decode_mma"
        assert txl.relattn_plan(B, 16, M, L, workspace_bytes=ws)[0] == want
        assert txl.relattn_plan(B, 16, M, L, workspace_bytes=0)[0] == want
    # An explicit tensor-core split needs its workspace.
    assert plan(16, 16, 1600, 128, 1728, 64, txl.BF16, 4, 0, ctypes.byref(k),
                ctypes.byref(n)) == WORKSPACE


L = txl.lib


def attn(**kw):
    a = dict(q=16, k=16, v=16, r=16, r_rows=8, u=16, vb=16, out=16, lse=None, B=1, H=1, M=4, L=4,
             dh=64, scale=0.125, dtype=txl.BF16, n_splits=1, ws=None, ws_bytes=0)
    a.update(kw)
    return L().txl_relattn_fwd(a["q"], a["k"], a["v"], a["r"], a["r_rows"], a["u"], a["vb"],
                               a["out"], a["lse"], a["B"], a["H"], a["M"], a["L"], a["dh"],
                               a["scale"], a["dtype"], a["n_splits"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), INVALID),
    (dict(out=None), INVALID),
    (dict(B=0), INVALID),
    (dict(L=0), INVALID),
    (dict(M=-1), INVALID),
    (dict(dtype=7), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(r_rows=7), SHAPE),
    (dict(dh=32), UNSUPPORTED),
    (dict(q=16 + 2), MISALIGNED),
    (dict(r=8), MISALIGNED),
    (dict(n_splits=2, M=1000, L=16, r_rows=1016), WORKSPACE),   # tensor-core path
    (dict(n_splits=12, M=2000, r_rows=2004), WORKSPACE),         # decode, beyond a cluster
    (dict(dtype=txl.F32, n_splits=2), UNSUPPORTED),
    (dict(dtype=txl.F32, k=2), MISALIGNED),
])
def test_relattn_validation(kw, want):
    assert attn(**kw) == want


def test_rel_pos_emb_validation():
    f = L().txl_rel_pos_emb
    assert f(None, 4, 8, txl.F32, None) == INVALID
    assert f(16, 0, 8, txl.F32, None) == INVALID
    assert f(16, 4, 7, txl.F32, None) == INVALID
    assert f(16, 4, 8, 3, None) == INVALID
    assert f(4, 4, 8, txl.F32, None) == MISALIGNED


def test_mem_validation_and_state():
    st = txl.MemState(0, 0, 8)
    # 16-byte rows are required: d=6 bf16 is 12 bytes.
    assert L().txl_mem_update(16, ctypes.byref(st), 16, 1, 2, 6, txl.BF16, None) == MISALIGNED
    bad = txl.MemState(9, 0, 8)
    assert L().txl_mem_update(16, ctypes.byref(bad), 16, 1, 2, 8, txl.BF16, None) == SHAPE
    bad = txl.MemState(0, 9, 8)
    assert L().txl_mem_concat(16, 16, ctypes.byref(bad), 16, 1, 2, 8, txl.BF16, None) == SHAPE
    # L = 0 and capacity 0 are no-ops that leave the state alone.
    st = txl.MemState(3, 5, 8)
    assert L().txl_mem_update(16, ctypes.byref(st), None, 1, 0, 8, txl.BF16, None) == OK
    assert (st.head, st.fill) == (3, 5)
    z = txl.MemState(0, 0, 0)
    assert L().txl_mem_update(None, ctypes.byref(z), 16, 1, 4, 8, txl.BF16, None) == OK
    assert (z.head, z.fill, z.capacity) == (0, 0, 0)
    assert L().txl_mem_concat(None, None, ctypes.byref(z), None, 1, 0, 8, txl.BF16, None) == OK


def test_python_binding_rejects_host_tensors():
    import torch
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        txl.relattn_fwd(q, q, q, q[0], q[0, 0, :1], q[0, 0, :1], 0, 0.125, out=q)


def _span(K, n):
    # keys of one decode key range: a whole number of 32-key chunks
    return ((K + n - 1) // n + 31) // 32 * 32


@pytest.mark.parametrize("B,H", [(1, 1), (1, 16), (2, 3), (8, 16), (64, 16)])
@pytest.mark.parametrize("M,L", [(0, 1), (1, 1), (127, 1), (300, 3), (3799, 1), (3800, 6), (511, 7),
                                 (4000, 8), (700, 9), (512, 512), (1600, 128), (3800, 128),
                                 (5000, 130)])
@pytest.mark.parametrize("n_splits", [0, 1, 2, 5, 9, 40])
def test_plan_splits_are_valid(B, H, M, L, n_splits):
    # Host logic only.  Whatever the request, the split the library picks must be
    # realisable: every decode key range owns keys (ranges of whole 32-key
    # chunks, at most one per 128 keys), tensor-core splits never exceed the
    # key tiles, and a split that needs partials needs the workspace.
    K = M + L
    ws = 1 << 34
    kernel, splits = txl.relattn_plan(B, H, M, L, n_splits=n_splits, workspace_bytes=ws)
    assert splits >= 1
    if kernel.startswith("decode"):
        assert L <= 8 and (kernel == "decode") == (L == 1)
        assert splits <= max(1, (K + 127) // 128)
        assert (splits - 1) * _span(K, splits) < K
        if n_splits:
            assert splits <= n_splits
    else:
        assert kernel == "tc"
        n_key_tiles = min(K - 1, M + L - 1) // 128 + 1
        assert splits <= n_key_tiles
        if n_splits:
            assert splits == min(n_splits, n_key_tiles)
        assert L > 8, "every segment of up to eight queries takes the decode kernel"
    if splits > 8 or (kernel == "tc" and splits > 1):
        # partials in the workspace: without one the call must refuse
        k, n = ctypes.c_int(0), ctypes.c_int(0)
        rc = txl.lib().txl_relattn_plan(B, H, M, L, K, 64, txl.BF16, n_splits, 0,
                                        ctypes.byref(k), ctypes.byref(n))
        if n_splits:
            assert rc == WORKSPACE
        else:
            assert rc == OK  # the automatic choice falls back to a split that fits


def attn_strided(kv_stride, **kw):
    a = dict(q=16, k=16, v=16, r=16, r_rows=8, u=16, vb=16, out=16, lse=None, B=1, H=1, M=4, L=4,
             dh=64, scale=0.125, dtype=txl.BF16, n_splits=1, ws=None, ws_bytes=0)
    a.update(kw)
    return L().txl_relattn_fwd_strided(a["q"], a["k"], a["v"], kv_stride, a["r"], a["r_rows"],
                                       a["u"], a["vb"], a["out"], a["lse"], a["B"], a["H"],
                                       a["M"], a["L"], a["dh"], a["scale"], a["dtype"],
                                       a["n_splits"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kv_stride,kw,want", [
    (0, {}, INVALID),                 # no plane stride given
    (8 * 64 - 8, {}, SHAPE),          # planes closer than K rows
    (8 * 64 + 4, {}, MISALIGNED),     # a plane would not start 16-byte aligned
    (8 * 64, dict(q=None), INVALID),  # the dense call's own checks still apply
    (8 * 64, dict(r_rows=7), SHAPE),
    (8 * 64, dict(dh=32), UNSUPPORTED),
    (4096, dict(n_splits=2, M=1000, L=16, r_rows=1016), SHAPE),
    (1016 * 64, dict(n_splits=2, M=1000, L=16, r_rows=1016), WORKSPACE),
])
def test_relattn_strided_validation(kv_stride, kw, want):
    assert attn_strided(kv_stride, **kw) == want


def test_kv_window_state_follows_the_memory():
    # Host arithmetic of the window (no kernel runs here): after each segment the
    # window holds the newest min(total, M) rows, and the rows of [memory ;
    # segment] it exposes stay inside the buffer.
    M, L, C = 100, 32, 2 * 100 + 32
    w = txl.KVWindow(0, 0, C, M)
    total = 0
    for _ in range(30):
        # what txl_kv_window_append does to the state: compaction when the
        # segment would not fit behind the memory
        if w.start + w.fill + L > C:
            w.start = 0
        assert w.start + w.fill + L <= C
        txl.kv_window_advance(w, L)
        total += L
        assert w.fill == min(total, M)
        assert 0 <= w.start and w.start + w.fill <= C


def test_kv_window_validation():
    w = txl.KVWindow(0, 0, 100, 50)
    # capacity below 2M + L
    assert L().txl_kv_window_append(16, ctypes.byref(w), 16, 4, 8, 64, txl.BF16, None) == SHAPE
    # a state whose window runs past the buffer, fill above M, negative start
    for bad in (txl.KVWindow(190, 20, 200, 50), txl.KVWindow(0, 60, 200, 50),
                txl.KVWindow(-1, 0, 200, 50)):
        assert L().txl_kv_window_append(16, ctypes.byref(bad), 16, 4, 8, 64, txl.BF16,
                                        None) == INVALID
        assert L().txl_kv_window_advance(ctypes.byref(bad), 8) == INVALID
    w = txl.KVWindow(0, 0, 200, 50)
    assert L().txl_kv_window_append(16, ctypes.byref(w), 16, 4, 8, 6, txl.BF16, None) == MISALIGNED
    assert L().txl_kv_window_append(16, ctypes.byref(w), 16, 4, 8, 64, 7, None) == INVALID
    # L = 0 appends nothing; advancing past the buffer's end is refused
    assert L().txl_kv_window_append(None, ctypes.byref(w), None, 4, 0, 64, txl.BF16, None) == OK
    w = txl.KVWindow(150, 50, 200, 50)
    assert L().txl_kv_window_advance(ctypes.byref(w), 8) == SHAPE
    assert (w.start, w.fill) == (150, 50)


def test_qkv_project_validation():
    # Host checks only (every case is refused or a no-op before any launch).
    w = txl.KVWindow(0, 0, 200, 50)
    st = txl.MemState(0, 0, 50)
    f = L().txl_qkv_project
    # null h / w / kv_buf / window, bad sizes, mem without its state
    assert f(None, 16, 2, 8, 64, 2, 64, 16, 16, ctypes.byref(w), None, None, None) == INVALID
    assert f(16, None, 2, 8, 64, 2, 64, 16, 16, ctypes.byref(w), None, None, None) == INVALID
    assert f(16, 16, 2, 8, 64, 2, 64, 16, None, ctypes.byref(w), None, None, None) == INVALID
    assert f(16, 16, 2, 8, 64, 2, 64, 16, 16, None, None, None, None) == INVALID
    assert f(16, 16, 0, 8, 64, 2, 64, 16, 16, ctypes.byref(w), None, None, None) == INVALID
    assert f(16, 16, 2, 8, 64, 2, 64, 16, 16, ctypes.byref(w), 16, None, None) == INVALID
    bad_st = txl.MemState(60, 0, 50)
    assert f(16, 16, 2, 8, 64, 2, 64, 16, 16, ctypes.byref(w), 16, ctypes.byref(bad_st),
             None) == INVALID
    assert f(16, 16, 2, 8, 64, 2, 64, 16, 16, ctypes.byref(txl.KVWindow(190, 20, 200, 50)), None,
             None, None) == INVALID
    # head width other than 64, window capacity below 2M + L, unaligned width / pointers
    assert f(16, 16, 2, 8, 64, 2, 32, 16, 16, ctypes.byref(w), None, None, None) == UNSUPPORTED
    assert f(16, 16, 2, 120, 64, 2, 64, 16, 16, ctypes.byref(w), None, None, None) == SHAPE
    assert f(16, 16, 2, 8, 60, 2, 64, 16, 16, ctypes.byref(w), None, None, None) == MISALIGNED
    assert f(8, 16, 2, 8, 64, 2, 64, 16, 16, ctypes.byref(w), None, None, None) == MISALIGNED
    assert f(16, 16, 2, 8, 64, 2, 64, 8, 16, ctypes.byref(w), None, None, None) == MISALIGNED
    # an empty segment changes nothing
    assert f(16, 16, 2, 0, 64, 2, 64, 16, 16, ctypes.byref(w), 16, ctypes.byref(st), None) == OK
    assert (w.start, w.fill, st.head, st.fill) == (0, 0, 0, 0)


def test_relattn_bwd_workspace_and_validation():
    # Host checks only: every case is refused before any launch.
    r256 = lambda x: (x + 255) // 256 * 256
    # three row chunks: row statistics, bias partials per (b, h, chunk or key
    # split: at least eight), g of every pair with rows of M + L = 200 rounded
    # up to 256
    rows = 3 * 5 * 130
    assert txl.bwd_workspace_size(3, 5, 130, 70) == (2 * r256(rows * 4) + r256(3 * 5 * 8 * 128 * 4) +
                                                     r256(rows * 256 * 4))
    # two row chunks: also the dq partials of up to eight key splits
    rows = 2 * 3 * 100
    assert txl.bwd_workspace_size(2, 3, 100, 50) == (2 * r256(rows * 4) + r256(2 * 3 * 8 * 128 * 4) +
                                                     r256(8 * rows * 64 * 4) + r256(rows * 192 * 4))
    assert txl.bwd_workspace_size(0, 5, 130, 70) == 0
    assert txl.bwd_workspace_size(3, 5, 130, -1) == 0
    f = L().txl_relattn_bwd
    p = 16  # a 16-byte aligned stand-in address (never dereferenced)
    ws_need = txl.bwd_workspace_size(2, 2, 8, 8)

    def call(**kw):
        a = dict(q=p, k=p, v=p, r=p, r_rows=16, u=p, vb=p, dout=p, dq=p, dk=p, dv=p, dr=p, du=p,
                 dvb=p, B=2, H=2, M=8, L=8, dh=64, scale=0.125, dtype=1, ws=256,
                 ws_bytes=ws_need)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["r"], a["r_rows"], a["u"], a["vb"], a["dout"], a["dq"],
                 a["dk"], a["dv"], a["dr"], a["du"], a["dvb"], a["B"], a["H"], a["M"], a["L"],
                 a["dh"], a["scale"], a["dtype"], a["ws"], a["ws_bytes"], None)

    assert call(q=None) == INVALID
    assert call(dr=None) == INVALID
    assert call(L=0) == INVALID
    assert call(M=-1) == INVALID
    assert call(dtype=7) == INVALID
    assert call(scale=float("nan")) == INVALID
    assert call(r_rows=15) == SHAPE
    assert call(dh=32) == UNSUPPORTED
    assert call(dtype=0) == UNSUPPORTED  # fp32 inputs: not supported by the backward
    assert call(k=8) == MISALIGNED
    assert call(dq=20) == MISALIGNED
    assert call(ws=None) == WORKSPACE
    assert call(ws_bytes=ws_need - 1) == WORKSPACE
    assert call(ws=272) == MISALIGNED
