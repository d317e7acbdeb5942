"""GPU parity of each kernel against the fp64 oracle, on seeded inputs that span
several tiles, ragged tails and the degenerate cases of the method.

"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context":
§3.3 (score, sinusoid R, masked softmax), §3.2 (memory), Appendix B (reversed
table and shift)."""

import math

import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_pos_gb300 as txl
from parity import (TOL_BF16, TOL_BF16_RMS, TOL_F32, compare, dev, heads_case, run_gpu,
                    run_oracle)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# device status word: the bounded-wait path gives up and reports
# ---------------------------------------------------------------------------

def test_barrier_wait_times_out_and_reports():
    dev()
    assert txl.device_status() == 0
    assert txl.debug_wait_timeout(20_000_000) == -6  # TXL_ERR_TIMEOUT after 20 ms
    assert txl.device_status() == 0  # the word was cleared


# ---------------------------------------------------------------------------
# sinusoid table (§3.3, Appendix B order)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K,d", [(1, 2), (32, 64), (1024, 512), (1728, 1024), (3928, 1024),
                                 (70000, 8), (300, 8192)])
def test_rel_pos_emb_matches_oracle(K, d):
    R = txl.rel_pos_emb(K, d, dtype=torch.float32, device=dev())
    want = oracle.reversed_table(oracle.sinusoid_table(K, d))
    # fp32 output: sincosf (about 1 ulp) on an angle reduced in double-float.
    compare(R.cpu().numpy(), want, 2e-6, what=f"R fp32 K={K} d={d}")
    Rb = txl.rel_pos_emb(K, d, dtype=torch.bfloat16, device=dev())
    # bf16 output: half a bf16 ulp of values <= 1 is 2^-9.
    compare(Rb.float().cpu().numpy(), want, 2.0 ** -8, what=f"R bf16 K={K} d={d}")


# ---------------------------------------------------------------------------
# memory ring buffer (§3.2): bit-exact against the oracle's trim of [m o h]
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,L,n_seg,dtype", [(100, 32, 9, torch.bfloat16), (20, 32, 4, torch.float32),
                                             (1600, 128, 15, torch.bfloat16), (7, 1, 12, torch.float32),
                                             (0, 16, 3, torch.bfloat16)])
def test_memory_ring_matches_oracle(M, L, n_seg, dtype):
    B, d = 3, 64
    g = torch.Generator().manual_seed(M * 31 + L)
    seq = torch.randn(B, n_seg * L, d, generator=g).to(dtype)
    mem = torch.zeros(B, max(M, 1), d, dtype=dtype, device=dev())[:, :M]
    mem = mem.contiguous()
    st = txl.MemState(0, 0, M)
    ref = np.zeros((B, 0, d))
    for s in range(n_seg):
        h = seq[:, s * L:(s + 1) * L].contiguous()
        hd = h.to(dev())
        ext = txl.mem_concat(mem, st, hd)
        want_ext = np.concatenate([ref, h.double().numpy()], axis=1)
        np.testing.assert_array_equal(ext.double().cpu().numpy(), want_ext)
        txl.mem_update(mem, st, hd)
        ref = oracle.memory_update(ref, h.double().numpy(), M)
        assert st.fill == ref.shape[1]
        assert st.head == ((s + 1) * L) % M if M else st.head == 0
    empty = torch.empty(B, 0, d, dtype=dtype, device=dev())
    np.testing.assert_array_equal(txl.mem_concat(mem, st, empty).double().cpu().numpy(), ref)
    assert txl.device_status() == 0


# ---------------------------------------------------------------------------
# attention, fp32 CUDA-core path
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,H,L,M", [(1, 1, 16, 16), (2, 3, 70, 45), (1, 2, 1, 0), (1, 1, 130, 0)])
def test_relattn_f32_matches_oracle(B, H, L, M):
    case = heads_case(B, H, L, M, seed=B * 100 + L + M, dtype=torch.float32)
    scale = 0.125
    out, lse = run_gpu(case, M, scale)
    want, want_lse = run_oracle(case, M, scale)
    compare(out.cpu().numpy(), want, TOL_F32, what="out f32")
    compare(lse.cpu().numpy(), want_lse, TOL_F32 * 10, what="lse f32")


# ---------------------------------------------------------------------------
# attention, bf16 tensor-core path
# ---------------------------------------------------------------------------

SHAPES = [
    # (B, H, L, M): full tiles, ragged query and key tails, empty memory,
    # one-token segments (decode-like), memory not a multiple of the tile.
    (1, 1, 128, 0),
    (1, 2, 128, 128),
    (2, 3, 100, 37),
    (1, 1, 1, 0),
    (1, 2, 1, 300),
    (2, 2, 200, 333),
    (1, 2, 16, 16),
    (1, 1, 300, 5),
    (3, 1, 257, 511),
    (1, 4, 128, 1600),
]


@pytest.mark.parametrize("B,H,L,M", SHAPES)
def test_relattn_bf16_matches_oracle(B, H, L, M):
    case = heads_case(B, H, L, M, seed=7 + B + 10 * H + L + M)
    scale = 1.0 / math.sqrt(64)
    out, lse = run_gpu(case, M, scale)
    want, want_lse = run_oracle(case, M, scale)
    compare(out.float().cpu().numpy(), want, TOL_BF16, TOL_BF16_RMS, what="out")
    compare(lse.cpu().numpy(), want_lse, TOL_BF16, what="lse")


@pytest.mark.parametrize("B,H,L,M", [(2, 2, 200, 333), (1, 2, 128, 1600)])
def test_relattn_bf16_sharp_softmax(B, H, L, M):
    # Larger operands make the softmax peaked, so a wrong relative index or
    # mask boundary changes which keys win.
    case = heads_case(B, H, L, M, seed=99 + L, std=2.5, bias_std=2.5)
    scale = 1.0 / math.sqrt(64)
    out, lse = run_gpu(case, M, scale)
    want, want_lse = run_oracle(case, M, scale)
    compare(out.float().cpu().numpy(), want, TOL_BF16, TOL_BF16_RMS, what="out sharp")
    compare(lse.cpu().numpy(), want_lse, 5e-2, what="lse sharp")


@pytest.mark.parametrize("n_splits", [2, 3, 5])
def test_relattn_bf16_key_splits(n_splits):
    B, H, L, M = 2, 2, 130, 900
    case = heads_case(B, H, L, M, seed=300 + n_splits)
    out, lse = run_gpu(case, M, 0.125, n_splits=n_splits)
    want, want_lse = run_oracle(case, M, 0.125)
    compare(out.float().cpu().numpy(), want, TOL_BF16, TOL_BF16_RMS, what=f"split {n_splits}")
    compare(lse.cpu().numpy(), want_lse, TOL_BF16, what=f"lse split {n_splits}")


# Launch shapes: one block per (batch, head, query tile) (n_splits 1) with
# more units than SMs, the automatic choice (0), and a key range split over
# seven blocks whose partial results are merged (7); plus many 1-row heads over
# a long memory.
@pytest.mark.parametrize("n_splits,B,H,L,M", [(1, 8, 16, 300, 100), (0, 8, 16, 300, 100),
                                              (1, 4, 40, 128, 200), (0, 4, 40, 128, 200),
                                              (7, 1, 2, 200, 900), (0, 3, 1, 1, 2000)])
def test_relattn_bf16_schedules(n_splits, B, H, L, M):
    case = heads_case(B, H, L, M, seed=700 + 13 * n_splits + L)
    out, lse = run_gpu(case, M, 0.125, n_splits=n_splits)
    want, want_lse = run_oracle(case, M, 0.125)
    what = f"schedule {n_splits} B{B} H{H} L{L} M{M}"
    compare(out.float().cpu().numpy(), want, TOL_BF16, TOL_BF16_RMS, what=what)
    compare(lse.cpu().numpy(), want_lse, TOL_BF16, what="lse " + what)


def test_relattn_bf16_merge_is_repeatable():
    # Split key ranges are merged in a fixed order: the result is bitwise stable.
    B, H, L, M = 2, 2, 130, 900
    case = heads_case(B, H, L, M, seed=77)
    a = run_gpu(case, M, 0.125, n_splits=5, want_lse=False)
    for _ in range(3):
        assert torch.equal(a, run_gpu(case, M, 0.125, n_splits=5, want_lse=False))


@pytest.mark.parametrize("L,M,n_splits", [(128, 8000, 0), (200, 8000, 5), (130, 12000, 1)])
def test_relattn_bf16_long_memory(L, M, n_splits):
    # Long memories (the evaluation of §3.2 with M in the thousands): 64 to 95 key
    # tiles per query tile, over one block, the automatic split and an explicit
    # one merged through the workspace.
    B, H = 1, 2
    case = heads_case(B, H, L, M, seed=800 + M // 1000 + L)
    out, lse = run_gpu(case, M, 0.125, n_splits=n_splits)
    want, want_lse = run_oracle(case, M, 0.125)
    what = f"long memory L={L} M={M} splits {n_splits}"
    compare(out.float().cpu().numpy(), want, TOL_BF16, TOL_BF16_RMS, what=what)
    compare(lse.cpu().numpy(), want_lse, TOL_BF16, what="lse " + what)


def test_relattn_bf16_longer_table():
    # A table built for a longer memory: only its last K rows are used.
    B, H, L, M = 1, 2, 128, 200
    case = heads_case(B, H, L, M, seed=5, extra_rows=700)
    out, _ = run_gpu(case, M, 0.125)
    want, _ = run_oracle(case, M, 0.125)
    compare(out.float().cpu().numpy(), want, TOL_BF16, TOL_BF16_RMS, what="long table")


def test_relattn_bf16_without_lse_and_repeatable():
    B, H, L, M = 2, 2, 128, 256
    case = heads_case(B, H, L, M, seed=8)
    a = run_gpu(case, M, 0.125, want_lse=False)
    b = run_gpu(case, M, 0.125, want_lse=False)
    assert torch.equal(a, b)  # deterministic: no atomics in the reduction
