"""txl_qkv_project on the GPU: one layer's projections of a segment ("Transformer-XL:
Attentive Language Models Beyond a Fixed-Length Context", §3.3 N-layer
summary: q = h W_q^T, k = h~ W_kE^T, v = h~ W_v^T, only the segment's rows new
when the memory's k and v are cached) written into q [B, H, L, 64] and the
rows behind the memory in the k / v window planes, with the memory update of
§3.2 in the same launch.

Checked against the unfused path on the same inputs: q, k, v against the fp64
products of the same bf16 operands (the kernel accumulates in fp32 and rounds
once to bf16: within one bf16 rounding plus fp32 summation, <= 1e-2 relative
to the row's scale); the window's memory rows, the ring, and both host states
bit for bit against txl_kv_window_append / txl_mem_update given the fused
kernel's own k and v."""

import numpy as np
import pytest
import torch

import transformer_xl_relative_pos_gb300 as txl
from parity import dev

pytestmark = pytest.mark.gpu


def _rand(g, *shape, std=1.0):
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def _case(B, L, d, H, M, C, start, fill, with_q, seed):
    g = torch.Generator().manual_seed(seed)
    n_out = 3 if with_q else 2
    h = _rand(g, B, L, d)
    w = _rand(g, n_out * H * 64, d, std=d ** -0.5)
    kv = _rand(g, 2 * B * H, C, 64)
    mem = _rand(g, B, M, d)
    return h, w, kv, mem


# (B, L, d_model, H, M, capacity, start, fill, with q, with the memory ring):
# ragged row tiles (B*L not a multiple of 128), L not dividing 128, output
# columns not a multiple of 256 (H = 3), d_model not a multiple of 64, a window
# that moves back to the front, an empty memory, no q, no ring.
CASES = [(2, 48, 128, 2, 100, 248, 0, 0, True, True),
         (3, 130, 512, 8, 64, 300, 36, 64, True, True),
         (2, 96, 200, 3, 80, 256, 90, 80, True, True),
         (1, 512, 512, 8, 512, 2048, 1024, 512, True, False),
         (2, 64, 256, 4, 128, 320, 0, 0, False, True)]


@pytest.mark.parametrize("B,L,d,H,M,C,start,fill,with_q,with_ring", CASES)
def test_qkv_project_matches_unfused_path(B, L, d, H, M, C, start, fill, with_q, with_ring):
    h, w, kv, mem = _case(B, L, d, H, M, C, start, fill, with_q, seed=B * 1000 + L + d)
    D = dev()
    h_d, w_d = h.to(D), w.to(D)
    kv_fused = kv.to(D)
    win = txl.KVWindow(start, fill, C, M)
    st = txl.MemState(7 % max(M, 1), min(fill, M), M)
    mem_fused = mem.to(D)
    q = torch.empty(B, H, L, 64, dtype=torch.bfloat16, device=D) if with_q else None
    txl.qkv_project(h_d, w_d, kv_fused, win, q=q, mem=mem_fused if with_ring else None,
                    mem_state=st if with_ring else None)
    torch.cuda.synchronize()
    assert txl.device_status() == 0

    # reference products in fp64 of the same bf16 operands, per output and head
    y = h.double().reshape(B * L, d) @ w.double().t()            # [B*L, n_out*H*64]
    n_out = 3 if with_q else 2
    y = y.reshape(B, L, n_out, H, 64).permute(2, 0, 3, 1, 4)   # [n_out, B, H, L, 64]
    scale = float(y.abs().max())
    outs = {}
    if with_q:
        outs["q"] = q.double().cpu()
    # the unfused path's window: the same start / compaction, the fused k, v as
    # the appended segment (so the memory rows and placement compare exactly)
    kv_seg = kv_fused.view(2 * B * H, C, 64)[:, win.start + win.fill:win.start + win.fill + L]
    outs["k"] = kv_seg[:B * H].double().cpu().reshape(B, H, L, 64)
    outs["v"] = kv_seg[B * H:].double().cpu().reshape(B, H, L, 64)
    for i, name in enumerate((["q"] if with_q else []) + ["k", "v"]):
        err = float((outs[name] - y[i]).abs().max())
        assert err <= 1e-2 * scale, f"{name}: max |err| {err:.3e} (scale {scale:.3e})"

    kv_ref = kv.to(D)
    win_ref = txl.KVWindow(start, fill, C, M)
    seg = kv_seg.contiguous()
    txl.kv_window_append(kv_ref, win_ref, seg)
    torch.cuda.synchronize()
    assert (win.start, win.fill) == (win_ref.start, win_ref.fill)
    assert torch.equal(kv_fused, kv_ref)   # memory rows moved or kept, segment rows placed
    if with_ring:
        mem_ref = mem.to(D)
        st_ref = txl.MemState(7 % max(M, 1), min(fill, M), M)
        txl.mem_update(mem_ref, st_ref, h_d)
        torch.cuda.synchronize()
        assert torch.equal(mem_fused, mem_ref)
        assert (st.head, st.fill) == (st_ref.head, st_ref.fill)
    assert txl.device_status() == 0


def test_qkv_project_repeatable():
    B, L, d, H, M, C = 2, 130, 512, 8, 64, 300
    h, w, kv, mem = _case(B, L, d, H, M, C, 0, 0, True, seed=5)
    D = dev()
    res = []
    for _ in range(2):
        kv_d = kv.to(D)
        q = torch.empty(B, H, L, 64, dtype=torch.bfloat16, device=D)
        txl.qkv_project(h.to(D), w.to(D), kv_d, txl.KVWindow(0, 0, C, M), q=q)
        torch.cuda.synchronize()
        res.append((q.clone(), kv_d.clone()))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
