"""Helpers shared by the GPU parity tests: build seeded inputs on the CPU, run
the CUDA path through the C ABI, run the fp64 oracle on the very same
(bf16- or fp32-rounded) values, and compare.

Tolerances (stated by the workload definitions):
  * fp32 path: max |GPU - oracle| <= 1e-5;
  * bf16 operands, fp32 accumulation: max |GPU - oracle| <= 2e-2 on O(1)
    outputs.  A second, tighter check bounds the error relative to the output
    RMS (<= 1e-2): a systematic mistake (a shifted relative index, a dropped
    bias) moves far more than that, while rounding of the bf16 output
    (2^-9 relative), of q+u / q+v and of P stays well inside it.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import txl_inputs
import transformer_xl_relative_pos_gb300 as txl
from transformer_xl_relative_pos_gb300 import model

TOL_F32 = 1e-5
TOL_BF16 = 2e-2
TOL_BF16_RMS = 1e-2


def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


def heads_case(B, H, L, M, seed, dtype=torch.bfloat16, std=1.0, bias_std=1.0, extra_rows=0):
    """Directly drawn operands (std-scaled), rounded once to ``dtype``.  With
    extra_rows > 0 the table gets that many leading rows (larger distances)."""
    d = txl_inputs.draw_heads(B, H, L, M, 64, seed, std=std, bias_std=bias_std)
    if extra_rows:
        g = torch.Generator().manual_seed(seed + 7)
        extra = torch.randn(H, extra_rows, 64, generator=g) * std
        d["r"] = torch.cat([extra, d["r"]], dim=1)
    return {k: v.to(dtype) for k, v in d.items()}


def layer_case(w: txl_inputs.Workload, sharp=False):
    """Operands of one layer built with the workload's recipe: states N(0,1),
    weights N(0,0.02), sinusoid table, projections in fp32 on the CPU, one
    rounding to the workload's dtype."""
    raw = txl_inputs.draw_layer(w, sharp=sharp)
    R_rev = torch.from_numpy(oracle.reversed_table(oracle.sinusoid_table(w.K, w.d_model))).float()
    dtype = torch.float32 if w.dtype == "f32" else torch.bfloat16
    q, k, v, r = model.attention_operands(raw["h_ext"], w.M, raw["W_q"], raw["W_kE"], raw["W_v"],
                                          raw["W_kR"], R_rev, w.H, dtype)
    return {"q": q, "k": k, "v": v, "r": r, "u": raw["u"].to(dtype),
            "v_bias": raw["v_bias"].to(dtype)}


def run_gpu(case, M, scale, n_splits=0, want_lse=True, workspace=True):
    d = dev()
    t = {k: v.to(d).contiguous() for k, v in case.items()}
    B, H, L, _ = t["q"].shape
    ws = None
    if workspace:
        nbytes = max(txl.workspace_size(B, H, L, 64, max(n_splits, 8)), 256)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=d)
    res = txl.relattn_fwd(t["q"], t["k"], t["v"], t["r"], t["u"], t["v_bias"], M, scale,
                          lse=True if want_lse else None, n_splits=n_splits, workspace=ws)
    torch.cuda.synchronize()
    assert txl.device_status() == 0, "a kernel reported a barrier time-out"
    return res


def run_oracle(case, M, scale, bh=None):
    K = case["k"].shape[2]
    rel = oracle.distance_table(case["r"][:, -K:].double().numpy())
    return oracle.relattn(case["q"], case["k"], case["v"], rel, case["u"], case["v_bias"],
                          M, case["q"].shape[2], scale, bh=bh)


def compare(got, want, tol, rms_tol=None, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite GPU output"
    err = np.abs(got - want)
    mx = float(err.max()) if err.size else 0.0
    assert mx <= tol, f"{what}: max |err| {mx:.3e} > {tol:.1e}"
    if rms_tol is not None and err.size:
        rel = math.sqrt(float((err ** 2).mean())) / max(math.sqrt(float((want ** 2).mean())), 1e-30)
        assert rel <= rms_tol, f"{what}: rms(err)/rms(out) {rel:.3e} > {rms_tol:.1e}"
    return mx
