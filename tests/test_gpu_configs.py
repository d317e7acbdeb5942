"""GPU parity on the five workloads, in the launch configuration the benchmark
times (automatic key splits with a workspace).

Small workloads are compared element by element; the full-size ones on
sampled (batch, head) slices that the oracle computes in seconds.  Inputs
follow each workload's recipe: states N(0,1), weights and biases N(0,0.02),
sinusoid table, one rounding to the workload's dtype."""

import math

import numpy as np
import pytest
import torch

import oracle
import txl_inputs
from parity import TOL_BF16, TOL_BF16_RMS, TOL_F32, compare, layer_case, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

W = txl_inputs.WORKLOADS


def test_c1_fp32_single_head_exact():
    w = W["c1_f32_L16_M16"]
    case = layer_case(w)
    scale = 1.0 / math.sqrt(w.dh)
    out, lse = run_gpu(case, w.M, scale)
    want, want_lse = run_oracle(case, w.M, scale)
    compare(out.cpu().numpy(), want, TOL_F32, what="c1 out")
    compare(lse.cpu().numpy(), want_lse, TOL_F32, what="c1 lse")


def sample_bh(B, H, n=8):
    BH = B * H
    picks = {0, BH - 1, H - 1, BH // 2, (BH // 3) | 1, H, BH - H, (2 * BH) // 3}
    return sorted(p for p in picks if 0 <= p < BH)[:n]


@pytest.mark.parametrize("name", ["c2_char_base_L512_M512", "c3_word_large_L128_M1600",
                                  "c4_long_mem_L128_M3800"])
@pytest.mark.parametrize("sharp", [False, True])
def test_full_size_sampled(name, sharp):
    w = W[name]
    case = layer_case(w, sharp=sharp)
    scale = 1.0 / math.sqrt(w.dh)
    out, lse = run_gpu(case, w.M, scale)
    bh = sample_bh(w.B, w.H)
    want, want_lse = run_oracle(case, w.M, scale, bh=bh)
    got = out.float().cpu().numpy()
    got_lse = lse.cpu().numpy()
    for p in bh:
        b, h = divmod(p, w.H)
        compare(got[b, h], want[b, h], TOL_BF16, TOL_BF16_RMS, what=f"{name} b={b} h={h}")
        compare(got_lse[b, h], want_lse[b, h], TOL_BF16, what=f"{name} lse b={b} h={h}")
    # Properties that hold at any size, over the whole output: finite, and each
    # output row inside the range spanned by the value rows it may see.
    assert np.isfinite(got).all() and np.isfinite(got_lse).all()
    v = case["v"].float()
    vmax = torch.cummax(v, dim=2).values[:, :, w.M:]   # visible keys j <= M + i
    vmin = torch.cummin(v, dim=2).values[:, :, w.M:]
    o = out.float().cpu()
    slack = 2e-2
    assert bool((o <= vmax + slack).all()) and bool((o >= vmin - slack).all())
