"""Pins of the oracle's backward (CPU only).

``oracle.relattn_bwd`` is the chain rule of the forward (training within a
segment, §3.2 of "Transformer-XL: Attentive Language Models Beyond a
Fixed-Length Context"; the score is §3.3's four-term A^rel).  It is tied to
things other than its own formulas:

  * central differences of the forward oracle (itself pinned by
    ``test_oracle_pins.py``) for every input: q, k, v, the by-distance table,
    u and v — including a batch of two (the table and biases are shared, so
    their gradients sum over the batch), an empty memory and one query;
  * with the table and both biases zero the score is plain content attention
    with the causal offset mask, so dq, dk, dv and du must equal the fp64
    backward of torch's scaled-dot-product attention (a library routine);
  * closed forms that hold for any input: the rows of P sum to one, so the
    value gradients sum to the summed output gradient and the key gradients
    sum to zero (a key-independent shift of the scores changes nothing).
"""

import numpy as np
import pytest

import oracle

SCALE = 0.5


def _draw(seed, B, H, M, L, dh, scale=1.0):
    rng = np.random.default_rng(seed)
    K = M + L
    f = lambda *s: rng.standard_normal(s) * scale
    return (f(B, H, L, dh), f(B, H, K, dh), f(B, H, K, dh), f(H, K, dh), f(H, dh), f(H, dh),
            rng.standard_normal((B, H, L, dh)))


def _loss(q, k, v, rel, u, vb, G, M, L):
    out, _ = oracle.relattn(q, k, v, rel, u, vb, M, L, SCALE)
    return float((out * G).sum())


@pytest.mark.parametrize("B,H,M,L,dh", [(1, 2, 3, 4, 4), (2, 1, 2, 3, 2), (1, 1, 0, 3, 4),
                                        (2, 2, 5, 1, 2)])
def test_gradients_match_central_differences(B, H, M, L, dh):
    q, k, v, rel, u, vb, G = _draw(11 + B + M, B, H, M, L, dh)
    grads = oracle.relattn_bwd(q, k, v, rel, u, vb, G, M, L, SCALE)
    inputs = [q, k, v, rel, u, vb]
    eps = 1e-6
    for pos, (x, g) in enumerate(zip(inputs, grads)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args_p = [t.copy() for t in inputs]
            args_m = [t.copy() for t in inputs]
            args_p[pos][idx] += eps
            args_m[pos][idx] -= eps
            fd[idx] = (_loss(*args_p, G, M, L) - _loss(*args_m, G, M, L)) / (2 * eps)
        # central differences of a smooth fp64 function: error ~eps^2 plus
        # rounding ~1e-16 / eps
        assert np.abs(fd - g).max() <= 1e-7 * max(1.0, np.abs(g).max()), pos


def test_reduces_to_sdpa_backward():
    torch = pytest.importorskip("torch")
    B, H, M, L, dh = 2, 3, 5, 4, 8
    q, k, v, _, _, _, G = _draw(5, B, H, M, L, dh)
    K = M + L
    rel = np.zeros((H, K, dh))
    u = np.zeros((H, dh))
    vb = np.zeros((H, dh))
    dq, dk, dv, drel, du, dvb = oracle.relattn_bwd(q, k, v, rel, u, vb, G, M, L, SCALE)

    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    tu = torch.zeros(H, 1, dh, dtype=torch.float64, requires_grad=True)
    i = torch.arange(L)[:, None]
    j = torch.arange(K)[None, :]
    keep = (j <= i + M)  # key j visible from query i: distance M + i - j >= 0
    out = torch.nn.functional.scaled_dot_product_attention(tq + tu, tk, tv, attn_mask=keep,
                                                           scale=SCALE)
    out.backward(torch.tensor(G, dtype=torch.float64))
    assert np.abs(tq.grad.numpy() - dq).max() < 1e-12
    assert np.abs(tk.grad.numpy() - dk).max() < 1e-12
    assert np.abs(tv.grad.numpy() - dv).max() < 1e-12
    assert np.abs(tu.grad.numpy()[:, 0, :] - du).max() < 1e-12
    assert np.abs(dvb).max() == 0.0  # term (d) is v . rel with rel = 0


@pytest.mark.parametrize("seed,M,L", [(1, 7, 5), (2, 0, 6), (3, 30, 2)])
def test_gradient_sums_closed_forms(seed, M, L):
    B, H, dh = 2, 2, 8
    q, k, v, rel, u, vb, G = _draw(seed, B, H, M, L, dh, scale=1.5)
    dq, dk, dv, drel, du, dvb = oracle.relattn_bwd(q, k, v, rel, u, vb, G, M, L, SCALE)
    # sum_j dv_j = sum_j sum_i P_ij dO_i = sum_i dO_i
    assert np.abs(dv.sum(axis=2) - G.sum(axis=2)).max() < 1e-10
    # sum_j dk_j = sum_i (sum_j g_ij) (q_i + u) = 0
    assert np.abs(dk.sum(axis=2)).max() < 1e-10
