"""Segment-level recurrence pins (CPU only).

"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
§3.2 (hidden states of the previous segments are cached and reused as an
extended context; the memory keeps the last M states) and the N-layer summary
of §3.3.  In a forward pass SG(.) is the identity, so a long sequence processed
segment by segment, with a memory that holds the whole prefix, must give the
same last-segment states as one pass over the concatenated sequence with causal
masking and relative distances measured in that sequence.
"""

import numpy as np
import pytest
import torch

import oracle


def small_stack(n_layer, d, H, dh, d_ff, vocab, seed):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: (torch.randn(*s, generator=g) * 0.3).double().numpy()
    layers = []
    for _ in range(n_layer):
        layers.append({
            "W_q": r(H * dh, d), "W_kE": r(H * dh, d), "W_v": r(H * dh, d), "W_kR": r(H * dh, d),
            "W_o": r(d, H * dh), "b_o": r(d), "W_1": r(d_ff, d), "b_1": r(d_ff),
            "W_2": r(d, d_ff), "b_2": r(d),
        })
    return {"emb": r(vocab, d), "u": r(H, dh), "v_bias": r(H, dh), "layers": layers}


@pytest.mark.parametrize("n_layer", [1, 3])
def test_stream_with_full_memory_equals_one_long_segment(n_layer):
    B, d, H, dh, d_ff, vocab, L, n_seg = 2, 16, 2, 8, 24, 11, 4, 3
    T = L * n_seg
    p = small_stack(n_layer, d, H, dh, d_ff, vocab, seed=9 + n_layer)
    g = torch.Generator().manual_seed(3)
    tokens = torch.randint(0, vocab, (B, T), generator=g).numpy()
    scale = dh ** -0.5
    M = T - L  # holds the whole prefix of the last segment
    mems = oracle.empty_memories(n_layer, B, d)
    for s in range(n_seg):
        h_seg, mems = oracle.segment_forward(tokens[:, s * L:(s + 1) * L], p["emb"], p["layers"],
                                             mems, p["u"], p["v_bias"], H, M, scale)
    h_full, _ = oracle.segment_forward(tokens, p["emb"], p["layers"],
                                       oracle.empty_memories(n_layer, B, d),
                                       p["u"], p["v_bias"], H, M, scale)
    np.testing.assert_allclose(h_seg, h_full[:, T - L:], rtol=1e-11, atol=1e-11)


def test_memory_keeps_last_M_states_oldest_first():
    B, d, L, M = 2, 3, 4, 6
    g = torch.Generator().manual_seed(21)
    seq = torch.randn(B, 5 * L, d, generator=g).double().numpy()
    mem = np.zeros((B, 0, d))
    for s in range(5):
        mem = oracle.memory_update(mem, seq[:, s * L:(s + 1) * L], M)
        end = (s + 1) * L
        np.testing.assert_array_equal(mem, seq[:, max(0, end - M):end])


def test_short_memory_equals_windowed_attention_over_the_sequence():
    # One layer, M smaller than the prefix: query g of the last segment sees
    # exactly the keys in [start - M, g] of the whole sequence.
    B, H, dh, d, L, n_seg, M = 1, 2, 4, 8, 3, 4, 5
    T = L * n_seg
    g = torch.Generator().manual_seed(31)
    seq = torch.randn(B, T, d, generator=g).double().numpy()
    W = [(torch.randn(H * dh, d, generator=g) * 0.4).double().numpy() for _ in range(4)]
    u = torch.randn(H, dh, generator=g).double().numpy()
    vb = torch.randn(H, dh, generator=g).double().numpy()
    mem = np.zeros((B, 0, d))
    for s in range(n_seg):
        h = seq[:, s * L:(s + 1) * L]
        q, k, v, rel = oracle.attention_inputs(h, mem, *W, H)
        out, _ = oracle.relattn(q, k, v, rel, u, vb, mem.shape[1], L, 0.5)
        mem = oracle.memory_update(mem, h, M)
    start = T - L
    # Same queries against the full sequence with keys before start-M removed
    # by an explicit score mask.
    qf, kf, vf, relf = oracle.attention_inputs(seq, np.zeros((B, 0, d)), *W, H)
    for h in range(H):
        for i in range(L):
            gq = start + i
            keys = range(start - M, gq + 1)
            logits = [0.5 * ((qf[0, h, gq] + u[h]) @ kf[0, h, j]
                             + (qf[0, h, gq] + vb[h]) @ relf[h, gq - j]) for j in keys]
            w = np.exp(np.array(logits) - max(logits))
            want = (w[:, None] * vf[0, h, list(keys)]).sum(0) / w.sum()
            np.testing.assert_allclose(out[0, h, i], want, rtol=1e-12, atol=1e-12)
