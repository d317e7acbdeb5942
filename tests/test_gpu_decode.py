"""GPU parity of the short-segment (decode) path against the fp64 oracle.

Generation feeds one or a few new tokens per step and attends to a long cached
memory ("Transformer-XL: Attentive Language Models Beyond a Fixed-Length
Context", §3.2 recurrence with a longer memory at evaluation, §3.3 score,
Appendix B reversed table).  txl_relattn_fwd takes every such call (bf16,
L <= 8) through a split-K decode kernel: for L >= 2 warp-level tensor-core
MMAs with q + u, q + v and the probabilities each carried as a bf16 value plus
its bf16 residual (about 2^-17 relative), fp32 accumulation and softmax; for
L = 1 fp32 arithmetic on the CUDA cores.  Either way the output differs from
the exact value by its bf16 rounding (2^-9 relative) and fp32 sums.
Tolerances: max |err| <= 1e-2 on O(1) outputs, rms(err)/rms(out) <= 4e-3,
log-sum-exp <= 1e-3.  L = 9 checks the hand-over to the 128-row tensor-core
kernel under the same tolerances.
"""

import math

import numpy as np
import pytest
import torch

import transformer_xl_relative_pos_gb300 as txl
from parity import compare, dev, heads_case, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

TOL = 1e-2
TOL_RMS = 4e-3
TOL_LSE = 1e-3


def check(case, M, n_splits=0, workspace=True, what=""):
    scale = 1.0 / math.sqrt(64)
    out, lse = run_gpu(case, M, scale, n_splits=n_splits, workspace=workspace)
    want, want_lse = run_oracle(case, M, scale)
    compare(out.float().cpu().numpy(), want, TOL, TOL_RMS, what=what)
    compare(lse.cpu().numpy(), want_lse, TOL_LSE, what="lse " + what)
    return out


# Query counts of the two decode kernels (1; 2..8) and past them, memories that
# end inside, at and just past a 128-key block, and none.
@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 6, 7, 8, 9])
@pytest.mark.parametrize("M", [0, 1, 127, 128, 300, 2000])
def test_decode_matches_oracle(L, M):
    B, H = 2, 3
    case = heads_case(B, H, L, M, seed=1000 + 17 * L + M)
    check(case, M, what=f"decode L={L} M={M}")


@pytest.mark.parametrize("n_splits,workspace", [(1, False), (0, False), (3, True), (7, True),
                                                (8, False), (9, True), (40, True)])
def test_decode_key_ranges(n_splits, workspace):
    # One block per head for all keys, the automatic choice without a
    # workspace, explicit splits merged inside a thread-block cluster (up to 8,
    # no workspace needed) or through the workspace (9 and more), and more
    # splits than 128-key chunks (capped).
    B, H, L, M = 2, 2, 3, 1500
    case = heads_case(B, H, L, M, seed=77 + n_splits)
    check(case, M, n_splits=n_splits, workspace=workspace, what=f"splits {n_splits}")


@pytest.mark.parametrize("L,n_splits", [(6, 1), (6, 5), (4, 0), (8, 1), (8, 3), (8, 11), (1, 11)])
def test_decode_long_segments_key_ranges(L, n_splits):
    # The largest decode segments (eight queries: a table window of 39 of the 40
    # rows a chunk copies), over one key range, ranges merged in a cluster and
    # through the workspace.
    B, H, M = 2, 3, 1100
    case = heads_case(B, H, L, M, seed=300 + 7 * L + n_splits)
    check(case, M, n_splits=n_splits, workspace=n_splits != 1, what=f"L={L} splits {n_splits}")


def test_decode_longer_table_and_sharp_scores():
    # A table built for a longer memory (only its last K rows are used) and
    # large scores, where the running-max rescale across chunks matters.
    B, H, L, M = 1, 2, 2, 900
    case = heads_case(B, H, L, M, seed=5, std=2.5, bias_std=2.5, extra_rows=333)
    check(case, M, what="long table, sharp")


@pytest.mark.parametrize("L", [1, 4, 8])
def test_decode_full_memory(L):
    # The long-memory evaluation shape (M = 3800) with one, four and eight new
    # tokens for a batch of 8 x 16 heads, in the launch the library picks;
    # every head is checked against the oracle.
    B, H, M = 8, 16, 3800
    case = heads_case(B, H, L, M, seed=11 + L)
    check(case, M, what=f"M=3800 L={L}")


@pytest.mark.parametrize("B,L,M", [(32, 4, 3800), (64, 6, 3800), (24, 1, 3800), (48, 8, 1600)])
def test_decode_large_batch_sampled_heads(B, L, M):
    # Many sequences: one key range per head and several waves of blocks; every
    # 29th head (of B x 16) is checked against the oracle.
    H = 16
    case = heads_case(B, H, L, M, seed=6000 + B + L)
    scale = 1.0 / math.sqrt(64)
    out, lse = run_gpu(case, M, scale)
    bh = list(range(0, B * H, 29))
    want_o, want_lse = run_oracle(case, M, scale, bh=bh)
    got, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
    for p in bh:
        b, h = divmod(p, H)
        compare(got[b, h], want_o[b, h], TOL, TOL_RMS, what=f"B={B} L={L} M={M} b={b} h={h}")
        compare(got_lse[b, h], want_lse[b, h], TOL_LSE, what=f"lse B={B} L={L} b={b} h={h}")


@pytest.mark.parametrize("L,M", [(8, 12000), (3, 20000), (1, 20000)])
def test_decode_very_long_memory(L, M):
    # One sequence against a memory far past the evaluation lengths: hundreds of
    # 32-key chunks per key range.
    B, H = 1, 4
    case = heads_case(B, H, L, M, seed=7000 + L)
    check(case, M, what=f"long memory L={L} M={M}")


def test_decode_repeatable():
    B, H, L, M = 2, 2, 3, 2000
    case = heads_case(B, H, L, M, seed=9)
    a = run_gpu(case, M, 0.125, want_lse=False)
    for _ in range(2):
        assert torch.equal(a, run_gpu(case, M, 0.125, want_lse=False))


@pytest.mark.parametrize("L,M", [(800, 0), (1, 799), (128, 672)])
def test_evaluation_speed_shapes(L, M):
    # The three ways of computing the attention of a window of 800 positions
    # compared by the evaluation-speed measurement (§4.5, Table 9): the vanilla
    # window from scratch, and state reuse with one or 128 new queries.
    B, H = 1, 2
    case = heads_case(B, H, L, M, seed=4500 + L)
    scale = 1.0 / math.sqrt(64)
    out, lse = run_gpu(case, M, scale)
    want, want_lse = run_oracle(case, M, scale)
    tol = TOL if L <= 8 else 2e-2  # the 128-row tensor-core kernel (L > 8) rounds P to bf16
    compare(out.float().cpu().numpy(), want, tol, 1e-2, what=f"window L={L} M={M}")
    compare(lse.cpu().numpy(), want_lse, 2e-2, what=f"lse window L={L} M={M}")


# Every segment of up to eight queries takes a decode kernel (one query the
# CUDA-core one, more the warp-MMA one), one sequence or many, short memory or
# long, with or without a workspace; nine queries take the 128-row tensor-core
# kernel.  An explicit split counts decode key ranges.
@pytest.mark.parametrize("B,L,M,want", [(1, 4, 8000, "decode_mma"), (1, 6, 3800, "decode_mma"),
                                        (8, 6, 3800, "decode_mma"), (2, 8, 800, "decode_mma"),
                                        (8, 1, 3800, "decode"), (1, 9, 1600, "tc")])
def test_short_segment_routing(B, L, M, want):
    H = 16
    ws_bytes = max(txl.workspace_size(B, H, L, 64, 64), 256)
    kernel, splits = txl.relattn_plan(B, H, M, L, workspace_bytes=ws_bytes)
    assert kernel == want, (B, L, M, kernel, splits)
    if want != "tc":
        assert txl.relattn_plan(B, H, M, L, n_splits=2, workspace_bytes=ws_bytes) == (want, 2)
        assert txl.relattn_plan(B, H, M, L, workspace_bytes=0)[0] == want
    case = heads_case(B, H, L, M, seed=4000 + 31 * L + M)
    d = dev()
    t = {k: v.to(d).contiguous() for k, v in case.items()}
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=d)
    scale = 1.0 / math.sqrt(64)
    out, lse = txl.relattn_fwd(t["q"], t["k"], t["v"], t["r"], t["u"], t["v_bias"], M, scale,
                               lse=True, workspace=ws)
    torch.cuda.synchronize()
    assert txl.device_status() == 0
    bh = list(range(0, B * H, 3))  # every third head keeps the oracle quick
    want_o, want_lse = run_oracle(case, M, scale, bh=bh)
    got, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
    for p in bh:
        b, h = divmod(p, H)
        compare(got[b, h], want_o[b, h], TOL, TOL_RMS, what=f"{kernel} B={B} L={L} M={M} h={h}")
        compare(got_lse[b, h], want_lse[b, h], TOL_LSE, what=f"lse {kernel} L={L} h={h}")


@pytest.mark.parametrize("B,H,M,L", [(1, 16, 3800, 1), (8, 16, 3800, 2), (2, 3, 300, 3), (64, 16, 3800, 6),
                                     (1, 16, 8000, 4), (4, 16, 12000, 8), (16, 16, 1600, 128),
                                     (8, 16, 3800, 128)])
@pytest.mark.parametrize("n_splits", [0, 3, 9])
def test_plan_on_device_is_realisable(B, H, M, L, n_splits):
    # The split chosen with this device's occupancy (not the host fallback):
    # decode ranges own keys and stay within one per 128 keys, tensor-core
    # splits within the key tiles.
    K = M + L
    kernel, splits = txl.relattn_plan(B, H, M, L, n_splits=n_splits, workspace_bytes=1 << 34)
    assert splits >= 1
    if kernel.startswith("decode"):
        span = ((K + splits - 1) // splits + 31) // 32 * 32
        assert splits <= max(1, (K + 127) // 128) and (splits - 1) * span < K
    else:
        assert splits <= min(K - 1, M + L - 1) // 128 + 1
