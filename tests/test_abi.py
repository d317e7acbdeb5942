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
    # Segments past six queries always take the tensor cores; the headline shape
    # (256 query tiles on 152 SMs) is not split.
    assert txl.relattn_plan(16, 16, 1600, 128, workspace_bytes=ws) == ("tc", 1)
    assert txl.relattn_plan(8, 16, 3800, 7, workspace_bytes=ws)[0] == "tc"
    # An explicit split of a short segment counts decode key ranges.
    assert txl.relattn_plan(8, 16, 3800, 6, n_splits=3, workspace_bytes=ws) == ("decode", 3)
    # The automatic choice for short segments follows the two kernels' estimates.
    assert txl.relattn_plan(8, 16, 3800, 1, workspace_bytes=ws)[0] == "decode"
    assert txl.relattn_plan(2, 16, 800, 6, workspace_bytes=ws)[0] == "decode"
    assert txl.relattn_plan(1, 16, 3800, 6, workspace_bytes=ws)[0] == "tc"
    # Without a workspace the tensor-core kernel cannot split one sequence's
    # keys, and the decode kernel (which merges inside a cluster) is cheaper.
    assert txl.relattn_plan(1, 16, 3800, 6, workspace_bytes=0)[0] == "decode"
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
                                 (512, 512), (1600, 128), (3800, 128), (5000, 130)])
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
    if kernel == "decode":
        assert L <= 6
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
        assert L > 6 or n_splits == 0, "an explicit split of a short segment means the decode kernel"
    if splits > 8 or (kernel == "tc" and splits > 1):
        # partials in the workspace: without one the call must refuse
        k, n = ctypes.c_int(0), ctypes.c_int(0)
        rc = txl.lib().txl_relattn_plan(B, H, M, L, K, 64, txl.BF16, n_splits, 0,
                                        ctypes.byref(k), ctypes.byref(n))
        if n_splits:
            assert rc == WORKSPACE
        else:
            assert rc == OK  # the automatic choice falls back to a split that fits
