"""k and v read in place from windows of larger buffers, and the memory kept as
such a window across segments.

"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
§3.2: the memory of the last M states is reused as extended context, [SG(m) o h]
(§3.3 summary).  txl_relattn_fwd_strided reads the K = M + L keys of each
(batch, head) plane from a window of a larger buffer (planes kv_stride elements
apart), and txl_kv_window_append / _advance keep a memory in such a window so
that nothing is concatenated before the attention.  Every row outside the windows
holds NaN: a kernel that read one would return NaN."""

import math

import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_pos_gb300 as txl
from parity import TOL_BF16, TOL_BF16_RMS, TOL_F32, compare, dev, heads_case, run_oracle

pytestmark = pytest.mark.gpu


def in_window(t, extra_front, extra_back):
    """t [B, H, K, dh] copied into a NaN-filled buffer [B*H, front + K + back, dh];
    returns the buffer and the [B, H, K, dh] window view."""
    B, H, K, dh = t.shape
    C = extra_front + K + extra_back
    buf = torch.full((B * H, C, dh), float("nan"), dtype=t.dtype, device=dev())
    view = buf.view(B, H, C, dh)[:, :, extra_front:extra_front + K]
    view.copy_(t.to(dev()))
    assert not view.is_contiguous()  # several planes: a strided window
    return buf, view


# (B, H, L, M, n_splits, dtype, kernel): tensor cores with a ragged segment and
# a key-range split, the two decode kernels (merged in a cluster, and through
# the workspace beyond one), the fp32 kernel.
CASES = [(2, 2, 130, 333, 0, torch.bfloat16, "tc"), (2, 2, 200, 900, 3, torch.bfloat16, "tc"),
         (2, 3, 3, 700, 0, torch.bfloat16, "decode_mma"), (1, 2, 5, 2000, 12, torch.bfloat16, "decode_mma"),
         (2, 3, 1, 700, 0, torch.bfloat16, "decode"), (1, 2, 1, 2000, 12, torch.bfloat16, "decode"),
         (1, 2, 16, 16, 1, torch.float32, "f32")]


@pytest.mark.parametrize("B,H,L,M,n_splits,dtype,kernel", CASES)
def test_relattn_strided_kv_matches_oracle_and_dense(B, H, L, M, n_splits, dtype, kernel):
    case = heads_case(B, H, L, M, seed=900 + L + M, dtype=dtype)
    d = dev()
    t = {k: v.to(d).contiguous() for k, v in case.items()}
    ws = torch.empty(max(txl.workspace_size(B, H, L, 64, max(n_splits, 16)), 256),
                     dtype=torch.uint8, device=d)
    assert txl.relattn_plan(B, H, M, L, dtype, n_splits=n_splits,
                            workspace_bytes=ws.numel())[0] == kernel
    _, kw = in_window(case["k"], 19, 45)
    _, vw = in_window(case["v"], 19, 45)
    out, lse = txl.relattn_fwd(t["q"], kw, vw, t["r"], t["u"], t["v_bias"], M, 0.125, lse=True,
                               n_splits=n_splits, workspace=ws)
    dense, dense_lse = txl.relattn_fwd(t["q"], t["k"], t["v"], t["r"], t["u"], t["v_bias"], M,
                                       0.125, lse=True, n_splits=n_splits, workspace=ws)
    torch.cuda.synchronize()
    assert txl.device_status() == 0
    # same kernel, same arithmetic: bit for bit what the dense call gives
    assert torch.equal(out, dense) and torch.equal(lse, dense_lse)
    want, want_lse = run_oracle(case, M, 0.125)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    compare(out.float().cpu().numpy(), want, tol, None if dtype == torch.float32 else TOL_BF16_RMS,
            what=f"strided {kernel}")
    compare(lse.cpu().numpy(), want_lse, tol * (10 if dtype == torch.float32 else 1), what="lse")


@pytest.mark.parametrize("M,L,extra", [(100, 32, 0), (100, 32, 77), (64, 150, 0), (0, 16, 5),
                                       (1600, 128, 0)])
def test_kv_window_holds_memory_and_segment(M, L, extra):
    # Through many segments (with capacity 2M + L the window moves back to the
    # buffer's front every few segments): the window exposes exactly [memory ;
    # segment] (bit for bit the oracle's trim of [m o h] followed by the new
    # rows), and after the advance the memory is the newest M rows.
    P, dh = 6, 64
    C = 2 * M + L + extra
    buf = torch.full((P, C, dh), float("nan"), dtype=torch.bfloat16, device=dev())
    w = txl.KVWindow(0, 0, C, M)
    ref = np.zeros((P, 0, dh))
    g = torch.Generator().manual_seed(M + 7 * L)
    starts = set()
    for s in range(3 * (2 * M // L + 3)):
        seg = torch.randn(P, L, dh, generator=g).to(torch.bfloat16)
        txl.kv_window_append(buf, w, seg.to(dev()))
        starts.add(w.start)
        got = buf[:, w.start:w.start + w.fill + L].double().cpu().numpy()
        np.testing.assert_array_equal(got, np.concatenate([ref, seg.double().numpy()], axis=1))
        txl.kv_window_advance(w, L)
        ref = oracle.memory_update(ref, seg.double().numpy(), M)
        assert w.fill == ref.shape[1]
        np.testing.assert_array_equal(buf[:, w.start:w.start + w.fill].double().cpu().numpy(), ref)
    if M > 0:
        # After an append the window started at the buffer's front (the first
        # segments, and again after moving back).  From the front, one more
        # segment fits behind the memory when 2L + M <= C, i.e. L <= M + extra;
        # otherwise every append moves the memory back first.
        assert 0 in starts
        assert (len(starts) > 1) == (L <= M + extra)
    assert txl.device_status() == 0


def test_attention_over_window_stream_equals_concatenated_memory():
    # A stream of segments: attention with k and v read in place from windows
    # equals, bit for bit, attention over the explicitly concatenated [memory ;
    # segment] kept in ring buffers (txl_mem_concat / txl_mem_update).
    B, H, L, M = 2, 2, 48, 100
    P = B * H
    C = 2 * M + L
    kbuf = torch.full((P, C, 64), float("nan"), dtype=torch.bfloat16, device=dev())
    vbuf = torch.full_like(kbuf, float("nan"))
    kw, vw = txl.KVWindow(0, 0, C, M), txl.KVWindow(0, 0, C, M)
    kring = torch.zeros(P, M, 64, dtype=torch.bfloat16, device=dev())
    vring = torch.zeros_like(kring)
    ks, vs = txl.MemState(0, 0, M), txl.MemState(0, 0, M)
    g = torch.Generator().manual_seed(3)
    # one table for the longest context; shorter ones use its last rows
    r = (torch.randn(H, M + L, 64, generator=g)).to(torch.bfloat16).to(dev())
    u = (torch.randn(H, 64, generator=g) * 0.5).to(torch.bfloat16).to(dev())
    vb = (torch.randn(H, 64, generator=g) * 0.5).to(torch.bfloat16).to(dev())
    for s in range(8):
        q = torch.randn(B, H, L, 64, generator=g).to(torch.bfloat16).to(dev())
        kn = torch.randn(P, L, 64, generator=g).to(torch.bfloat16).to(dev())
        vn = torch.randn(P, L, 64, generator=g).to(torch.bfloat16).to(dev())
        m_cur = ks.fill
        txl.kv_window_append(kbuf, kw, kn)
        txl.kv_window_append(vbuf, vw, vn)
        got = txl.relattn_fwd(q, txl.kv_window_view(kbuf, kw, L, B, H),
                              txl.kv_window_view(vbuf, vw, L, B, H), r, u, vb, m_cur, 0.125)
        kx = txl.mem_concat(kring, ks, kn).view(B, H, m_cur + L, 64)
        vx = txl.mem_concat(vring, vs, vn).view(B, H, m_cur + L, 64)
        want = txl.relattn_fwd(q, kx, vx, r, u, vb, m_cur, 0.125)
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"segment {s}"
        txl.kv_window_advance(kw, L)
        txl.kv_window_advance(vw, L)
        txl.mem_update(kring, ks, kn)
        txl.mem_update(vring, vs, vn)
    assert txl.device_status() == 0
