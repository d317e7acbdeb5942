"""GPU parity of the backward (``txl_relattn_bwd``) against the fp64 oracle.

"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context": §3.2
(training backpropagates within a segment; the memory is SG(m), its projected
k and v still receive gradients), §3.3 (the four-term score), Appendix B (the
reversed table: the table gradient comes back in the same row order).

Tolerance.  Inputs are bf16 and reach both sides unrounded further; the CUDA
path accumulates in fp32 (scores over 64 dimensions, the statistics and the
gradient sums over up to a few thousand keys or rows), so its error is a few
fp32 roundings of the largest terms: bounded here by 2e-4 of each gradient's
largest entry, with the RMS of the error under 2e-5 of it.  A wrong index, a
dropped term or a transposed operand moves entries by O(1) of that scale.
"""

import numpy as np
import pytest
import torch

import oracle
import transformer_xl_relative_pos_gb300 as txl
from parity import dev, heads_case

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dr", "du", "dv_bias")


def _oracle_grads(case, dout, M, scale):
    K = case["k"].shape[2]
    L = case["q"].shape[2]
    rel = oracle.distance_table(case["r"][:, -K:].double().numpy())
    return oracle.relattn_bwd(case["q"], case["k"], case["v"], rel, case["u"], case["v_bias"],
                              dout, M, L, scale)


def _gpu_grads(case, dout, M, scale):
    d = dev()
    t = {k: v.to(d).contiguous() for k, v in case.items()}
    g = txl.relattn_bwd(t["q"], t["k"], t["v"], t["r"], t["u"], t["v_bias"],
                        dout.to(d).contiguous(), M, scale)
    torch.cuda.synchronize()
    assert txl.device_status() == 0
    return [x.cpu().numpy().astype(np.float64) for x in g]


def _check(got, want, K, what):
    dq, dk, dv, dr, du, dvb = got
    r_rows = dr.shape[1]
    # the table gradient comes back in the reversed row order; rows of
    # distances >= K are zero
    dr_by_distance = np.flip(dr[:, r_rows - K:], axis=1)
    assert np.all(dr[:, :r_rows - K] == 0.0), f"{what}: rows past the last distance"
    for name, g, w in zip(NAMES, (dq, dk, dv, dr_by_distance, du, dvb), want):
        scale = max(np.abs(w).max(), 1e-30)
        err = np.abs(g - w)
        assert err.max() <= 2e-4 * scale, f"{what} {name}: max err {err.max():.3e} of {scale:.3e}"
        assert np.sqrt((err ** 2).mean()) <= 2e-5 * scale, f"{what} {name}: rms err"


# (B, H, L, M, extra table rows, input std): several tiles and ragged tails in
# every direction (64-row chunks, 64-key tiles, 64-distance tiles), no memory,
# one query, a table longer than the keys, a peaked softmax.  Segments of up to
# 128 rows run the two-chunk kernels over key splits: one split when the keys
# fit one tile (1, 2, 40, 20) or when B*H blocks already fill whole waves of a
# 152-SM part (8, 19, 64, 64); two or more otherwise.
CASES = [
    (2, 3, 50, 70, 0, 1.0),
    (1, 2, 130, 130, 0, 1.0),
    (2, 2, 65, 0, 0, 1.0),
    (1, 2, 1, 200, 0, 1.0),
    (2, 1, 64, 64, 0, 1.0),
    (1, 2, 40, 100, 37, 1.0),
    (2, 2, 96, 150, 0, 3.0),
    (1, 1, 300, 200, 64, 1.0),
    (1, 2, 40, 20, 0, 1.0),
    (8, 19, 64, 64, 0, 1.0),
]


@pytest.mark.parametrize("B,H,L,M,extra,std", CASES)
def test_backward_matches_oracle(B, H, L, M, extra, std):
    case = heads_case(B, H, L, M, seed=B * 131 + L * 7 + M, std=std, bias_std=0.5 * std,
                      extra_rows=extra)
    g = torch.Generator().manual_seed(L + 3 * M)
    dout = torch.randn(B, H, L, 64, generator=g).to(torch.bfloat16)
    scale = 0.125
    got = _gpu_grads(case, dout, M, scale)
    want = _oracle_grads(case, dout, M, scale)
    _check(got, want, M + L, f"B{B} H{H} L{L} M{M}")


def test_backward_headline_size_sampled_heads():
    """The headline workload's sizes (B=16, H=16, L=128, M=1600); the oracle
    recomputes two heads (every batch row, so their table and bias gradients
    are complete)."""
    B, H, L, M = 16, 16, 128, 1600
    case = heads_case(B, H, L, M, seed=99, std=0.6, bias_std=0.3)
    g = torch.Generator().manual_seed(5)
    dout = torch.randn(B, H, L, 64, generator=g).to(torch.bfloat16)
    scale = 0.125
    got = _gpu_grads(case, dout, M, scale)
    heads = [3, 14]
    sub = {k: (v[:, heads] if k in ("q", "k", "v") else v[heads]) for k, v in case.items()}
    want = _oracle_grads(sub, dout[:, heads], M, scale)
    dq, dk, dv, dr, du, dvb = got
    got_sub = [dq[:, heads], dk[:, heads], dv[:, heads], dr[heads], du[heads], dvb[heads]]
    _check(got_sub, want, M + L, "headline heads 3, 14")


def test_backward_long_memory_seven_splits_sampled_heads():
    """B=8, H=16, L=128, M=3800 (a long memory): 128 (batch, head) blocks, so
    the key range is split seven ways on a 152-SM part; the oracle recomputes
    two heads over every batch row."""
    B, H, L, M = 8, 16, 128, 3800
    case = heads_case(B, H, L, M, seed=41, std=0.6, bias_std=0.3)
    g = torch.Generator().manual_seed(8)
    dout = torch.randn(B, H, L, 64, generator=g).to(torch.bfloat16)
    scale = 0.125
    got = _gpu_grads(case, dout, M, scale)
    heads = [5, 11]
    sub = {k: (v[:, heads] if k in ("q", "k", "v") else v[heads]) for k, v in case.items()}
    want = _oracle_grads(sub, dout[:, heads], M, scale)
    dq, dk, dv, dr, du, dvb = got
    got_sub = [dq[:, heads], dk[:, heads], dv[:, heads], dr[heads], du[heads], dvb[heads]]
    _check(got_sub, want, M + L, "long memory heads 5, 11")


def test_backward_repeats_bit_for_bit():
    case = heads_case(2, 2, 100, 300, seed=7)
    dout = torch.randn(2, 2, 100, 64, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    a = _gpu_grads(case, dout, 300, 0.125)
    b = _gpu_grads(case, dout, 300, 0.125)
    for x, y, name in zip(a, b, NAMES):
        assert np.array_equal(x, y), name


def test_backward_rejects_bad_arguments():
    d = dev()
    case = {k: v.to(d) for k, v in heads_case(1, 1, 8, 8, seed=3).items()}
    dout = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device=d)
    small_ws = torch.empty(16, dtype=torch.uint8, device=d)
    with pytest.raises(txl.TxlError):
        txl.relattn_bwd(case["q"], case["k"], case["v"], case["r"], case["u"], case["v_bias"],
                        dout, 8, 0.125, workspace=small_ws)
    with pytest.raises(txl.TxlError):  # table shorter than the keys
        txl.relattn_bwd(case["q"], case["k"], case["v"], case["r"][:, 1:].contiguous(),
                        case["u"], case["v_bias"], dout, 8, 0.125)
