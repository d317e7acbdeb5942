"""Seeded synthetic inputs for the Transformer-XL relative-attention workloads.

This module is shared by the fp64 oracle side and the CUDA side of the tests and
of ``bench.py``.  It holds shapes and random draws only: no arithmetic of the
method (no projection, no positional table, no score, no softmax) lives here.

Every tensor is drawn on the CPU with ``torch.Generator().manual_seed(seed)`` in
fp32, in a fixed order, so that both sides see identical values.

Distributions (the evaluation shapes of "Transformer-XL: Attentive Language
Models Beyond a Fixed-Length Context", §4.1 and Table 9, stand-ins for the
WikiText-103 / enwik8 data, which are not used):
  * hidden and memory states ~ N(0, 1)
  * W_q, W_kE, W_v, W_kR and the global biases u, v ~ N(0, 0.02)
  * the "sharp" variant draws weights ~ N(0, 1/d_model) and u, v ~ N(0, 1), so
    that the softmax is peaked and the relative shift and the mask decide the
    result.
"""

from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention workload: batch B, heads H, head size dh, segment length L,
    memory length M (keys K = M + L, memory rows first), model width d_model."""

    name: str
    B: int
    H: int
    dh: int
    L: int
    M: int
    d_model: int
    dtype: str  # "f32" or "bf16": the element type the kernel receives
    seed: int
    d_ff: int = 0
    n_layer: int = 1
    n_seg: int = 1
    vocab: int = 0

    @property
    def K(self) -> int:
        return self.M + self.L

    def flops(self) -> float:
        """Nominal forward FLOPs of one attention call: 6*L*K*dh per head
        (three contractions: content scores, position scores, P.V)."""
        return 6.0 * self.L * self.K * self.dh * self.B * self.H


# The five workloads.  Names describe the shape; seeds are fixed.
WORKLOADS = {
    "c1_f32_L16_M16": Workload("c1_f32_L16_M16", B=1, H=1, dh=64, L=16, M=16,
                               d_model=64, dtype="f32", seed=0),
    "c2_char_base_L512_M512": Workload("c2_char_base_L512_M512", B=16, H=8, dh=64,
                                       L=512, M=512, d_model=512, dtype="bf16", seed=1),
    "c3_word_large_L128_M1600": Workload("c3_word_large_L128_M1600", B=16, H=16, dh=64,
                                         L=128, M=1600, d_model=1024, dtype="bf16", seed=2),
    "c4_long_mem_L128_M3800": Workload("c4_long_mem_L128_M3800", B=8, H=16, dh=64,
                                       L=128, M=3800, d_model=1024, dtype="bf16", seed=3),
    "c5_stack12_L512_M512": Workload("c5_stack12_L512_M512", B=16, H=8, dh=64, L=512,
                                     M=512, d_model=512, dtype="bf16", seed=4, d_ff=2048,
                                     n_layer=12, n_seg=16, vocab=204),
}

HEADLINE = "c3_word_large_L128_M1600"


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def draw_layer(w: Workload, sharp: bool = False, seed: int | None = None) -> dict:
    """Raw draws for one attention layer over an extended context of K rows.

    Returns fp32 CPU tensors:
      h_ext [B, K, d_model]  memory states (rows 0..M-1) then the segment (rows M..K-1)
      W_q, W_kE, W_v, W_kR [H*dh, d_model]
      u, v_bias [H, dh]
    """
    g = _gen(w.seed if seed is None else seed)
    d, hd = w.d_model, w.H * w.dh
    wstd = (1.0 / d) ** 0.5 if sharp else 0.02
    bstd = 1.0 if sharp else 0.02
    out = {"h_ext": torch.randn(w.B, w.K, d, generator=g)}
    for name in ("W_q", "W_kE", "W_v", "W_kR"):
        out[name] = torch.randn(hd, d, generator=g) * wstd
    out["u"] = torch.randn(w.H, w.dh, generator=g) * bstd
    out["v_bias"] = torch.randn(w.H, w.dh, generator=g) * bstd
    return out


def draw_heads(B: int, H: int, L: int, M: int, dh: int, seed: int, std: float = 1.0,
               bias_std: float = 1.0) -> dict:
    """Directly drawn per-head operands for small parity and edge cases.

    q [B,H,L,dh], k/v [B,H,K,dh], r [H,K,dh], u/v_bias [H,dh]; fp32 CPU."""
    g = _gen(seed)
    K = M + L
    return {
        "q": torch.randn(B, H, L, dh, generator=g) * std,
        "k": torch.randn(B, H, K, dh, generator=g) * std,
        "v": torch.randn(B, H, K, dh, generator=g),
        "r": torch.randn(H, K, dh, generator=g) * std,
        "u": torch.randn(H, dh, generator=g) * bias_std,
        "v_bias": torch.randn(H, dh, generator=g) * bias_std,
    }


def draw_stack(w: Workload) -> dict:
    """Raw draws for the streaming N-layer stack: token stream, embeddings and
    per-layer weights (all ~N(0, 0.02)); one u, v shared by all layers.

    tokens [n_seg, B, L] int64 uniform over the vocabulary."""
    g = _gen(w.seed)
    d, hd, f = w.d_model, w.H * w.dh, w.d_ff
    s = 0.02
    out = {
        "tokens": torch.randint(0, w.vocab, (w.n_seg, w.B, w.L), generator=g),
        "emb": torch.randn(w.vocab, d, generator=g) * s,
        "u": torch.randn(w.H, w.dh, generator=g) * s,
        "v_bias": torch.randn(w.H, w.dh, generator=g) * s,
        "layers": [],
    }
    for _ in range(w.n_layer):
        lay = {}
        for name in ("W_q", "W_kE", "W_v", "W_kR"):
            lay[name] = torch.randn(hd, d, generator=g) * s
        lay["W_o"] = torch.randn(d, hd, generator=g) * s
        lay["b_o"] = torch.randn(d, generator=g) * s
        lay["W_1"] = torch.randn(f, d, generator=g) * s
        lay["b_1"] = torch.randn(f, generator=g) * s
        lay["W_2"] = torch.randn(d, f, generator=g) * s
        lay["b_2"] = torch.randn(d, generator=g) * s
        out["layers"].append(lay)
    return out
