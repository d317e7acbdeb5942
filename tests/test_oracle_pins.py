"""Pins of the fp64 oracle to what the pages and mathematics fix (CPU only).

Each test ties the oracle to something other than itself:
  * hand-worked examples of the §3.3 score (tests/golden/hand_worked.json);
  * closed forms and identities of the sinusoid table;
  * the algebraic identity between the four terms (a)-(d) and the compact
    (q+u).k + (q+v).W_kR R grouping;
  * the reduction to ordinary causal attention (torch's scaled_dot_product_attention);
  * Appendix B's shifted-matrix relation;
  * segment-level recurrence = attention over the explicit extended context;
  * an independently written pure-Python brute force on tiny shapes;
  * softmax invariants (rows sum to one, masked keys get zero weight).

"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context" is
cited by section below.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import txl_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def rand_heads(B, H, L, M, dh, seed, std=1.0):
    d = txl_inputs.draw_heads(B, H, L, M, dh, seed, std=std)
    return {k: v.double().numpy() for k, v in d.items()}


# ---------------------------------------------------------------------------
# Hand-worked examples (§3.3 A^rel; masked softmax)
# ---------------------------------------------------------------------------

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_terms_and_output(case):
    M, L, scale = case["M"], case["L"], case["scale"]
    q = np.array(case["q"])[None, None]
    k = np.array(case["k"])[None, None]
    v = np.array(case["v"])[None, None]
    rel = np.array(case["rel_by_distance"])[None]
    u = np.array(case["u"])[None]
    vb = np.array(case["v_bias"])[None]
    ta, tb, tc, td, valid = oracle.score_terms(q[0, 0], k[0, 0], rel[0], u[0], vb[0], M, L)
    for key, t in case["terms_by_hand"].items():
        parts = key.split("_")
        i, j = int(parts[0][3:]), int(parts[1][3:])
        assert valid[i, j]
        assert (ta[i, j], tb[i, j], tc[i, j], td[i, j]) == (t["a"], t["b"], t["c"], t["d"])
    out, lse = oracle.relattn(q, k, v, rel, u, vb, M, L, scale)
    for i, row in enumerate(case["scaled_logits"]):
        vis = [(j, x) for j, x in enumerate(row) if x is not None]
        for j, x in enumerate(row):
            assert bool(valid[i, j]) == (x is not None)
        top = max(x for _, x in vis)
        z = sum(math.exp(x - top) for _, x in vis)
        want = sum(math.exp(x - top) * case["v"][j][0] for j, x in vis) / z
        assert out[0, 0, i, 0] == pytest.approx(want, rel=1e-14, abs=1e-14)
        assert lse[0, 0, i] == pytest.approx(top + math.log(z), rel=1e-14)
    if case["name"] == "M1_L1":
        p = 1.0 / (1.0 + math.exp(5.75))
        assert out[0, 0, 0, 0] == pytest.approx(7.0 - 2.0 * p, rel=1e-14)
    if case["name"] == "M0_L1":
        assert out[0, 0, 0, 0] == case["v"][0][0]


def test_single_visible_key_returns_value_row():
    # L=1, M=0: the only visible key is the query's own position.
    d = rand_heads(2, 3, 1, 0, 8, seed=11)
    out, _ = oracle.relattn(d["q"], d["k"], d["v"], d["r"], d["u"], d["v_bias"], 0, 1, 0.3)
    np.testing.assert_array_equal(out[:, :, 0, :], d["v"][:, :, 0, :])


def test_first_query_of_empty_memory_sees_only_itself():
    # M=0: query 0 sees key 0 only, whatever L is (causal within the segment).
    d = rand_heads(1, 2, 5, 0, 4, seed=12)
    out, _ = oracle.relattn(d["q"], d["k"], d["v"], d["r"], d["u"], d["v_bias"], 0, 5, 0.5)
    np.testing.assert_array_equal(out[:, :, 0, :], d["v"][:, :, 0, :])


# ---------------------------------------------------------------------------
# Sinusoid table (§3.3: R is the sinusoid encoding matrix, row p = distance p)
# ---------------------------------------------------------------------------

def test_sinusoid_row_zero_and_unit_pairs():
    R = oracle.sinusoid_table(50, 16)
    np.testing.assert_array_equal(R[0], np.tile([0.0, 1.0], 8))
    pair_norm = R[:, 0::2] ** 2 + R[:, 1::2] ** 2
    np.testing.assert_allclose(pair_norm, 1.0, atol=1e-15)


def test_sinusoid_closed_form_frequencies():
    # d = 2: one pair at frequency 10000^0 = 1 -> [sin p, cos p].
    R2 = oracle.sinusoid_table(40, 2)
    for p in range(40):
        assert R2[p, 0] == pytest.approx(math.sin(p), abs=1e-15)
        assert R2[p, 1] == pytest.approx(math.cos(p), abs=1e-15)
    # d = 4: the second pair runs at 10000^(-2/4) = 0.01.
    R4 = oracle.sinusoid_table(40, 4)
    for p in range(40):
        assert R4[p, 2] == pytest.approx(math.sin(0.01 * p), abs=1e-15)
        assert R4[p, 3] == pytest.approx(math.cos(0.01 * p), abs=1e-15)


def test_sinusoid_rotation_and_relative_kernel():
    # Each (sin, cos) pair rotates by w_k per step: angle addition with row 1.
    d = 64
    R = oracle.sinusoid_table(300, d)
    s1, c1 = R[1, 0::2], R[1, 1::2]
    s, c = R[:-1, 0::2], R[:-1, 1::2]
    np.testing.assert_allclose(R[1:, 0::2], s * c1 + c * s1, atol=1e-12)
    np.testing.assert_allclose(R[1:, 1::2], c * c1 - s * s1, atol=1e-12)
    # R_p . R_q = sum_k cos((p - q) w_k): depends on p - q only.
    G = R @ R.T
    for p, qq in [(10, 3), (250, 243), (17, 17), (0, 7)]:
        assert G[p, qq] == pytest.approx(R[abs(p - qq), 1::2].sum(), abs=1e-11)


def test_sinusoid_rejects_odd_width():
    with pytest.raises(ValueError):
        oracle.sinusoid_table(4, 7)


# ---------------------------------------------------------------------------
# §3.3: four terms == compact grouping; Appendix B shift relation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,L,dh", [(0, 5, 8), (7, 4, 16), (13, 9, 64)])
def test_four_terms_equal_compact_form(M, L, dh):
    d = rand_heads(1, 1, L, M, dh, seed=100 + M)
    q, k, rel, u, vb = d["q"][0, 0], d["k"][0, 0], d["r"][0], d["u"][0], d["v_bias"][0]
    ta, tb, tc, td, valid = oracle.score_terms(q, k, rel, u, vb, M, L)
    K = M + L
    ii, jj = np.meshgrid(np.arange(L), np.arange(K), indexing="ij")
    dist = M + ii - jj
    content = (q + u) @ k.T
    pos = np.einsum("it,ijt->ij", q + vb, rel[np.clip(dist, 0, K - 1)])
    compact = np.where(dist >= 0, content + pos, 0.0)
    np.testing.assert_allclose(ta + tb + tc + td, compact, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(valid, dist >= 0)


@pytest.mark.parametrize("M,L", [(0, 6), (5, 3), (9, 9), (20, 7)])
def test_appendix_b_shift_gives_term_b(M, L):
    d = rand_heads(1, 1, L, M, 8, seed=200 + M)
    q, k, rel = d["q"][0, 0], d["k"][0, 0], d["r"][0]
    _, tb, _, _, valid = oracle.score_terms(q, k, rel, d["u"][0], d["v_bias"][0], M, L)
    Bm = oracle.appendix_b_position_term(q, rel, M, L)
    np.testing.assert_allclose(Bm, np.where(valid, tb, 0.0), rtol=1e-13, atol=1e-13)
    # Appendix B's reversed Q: row k = W_kR R_{M+L-1-k}.
    Q = oracle.reversed_table(rel)
    np.testing.assert_array_equal(Q[0], rel[M + L - 1])
    np.testing.assert_array_equal(Q[-1], rel[0])


# ---------------------------------------------------------------------------
# Reduction to ordinary causal attention (u = v = 0, W_kR = 0)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,L", [(0, 7), (6, 5), (33, 17)])
def test_reduces_to_causal_sdpa(M, L):
    B, H, dh = 2, 3, 16
    d = rand_heads(B, H, L, M, dh, seed=300 + L)
    zeros_h = np.zeros((H, dh))
    rel0 = np.zeros((H, M + L, dh))
    scale = dh ** -0.5
    out, _ = oracle.relattn(d["q"], d["k"], d["v"], rel0, zeros_h, zeros_h, M, L, scale)
    ii = torch.arange(L)[:, None]
    jj = torch.arange(M + L)[None, :]
    mask = jj <= ii + M
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(d["q"]), torch.from_numpy(d["k"]), torch.from_numpy(d["v"]),
        attn_mask=mask, scale=scale)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_only_global_content_bias_matches_sdpa_with_shifted_queries():
    # With W_kR = 0 the score is (q+u).k: SDPA on q+u.
    B, H, L, M, dh = 1, 2, 6, 4, 8
    d = rand_heads(B, H, L, M, dh, seed=333)
    rel0 = np.zeros((H, M + L, dh))
    out, _ = oracle.relattn(d["q"], d["k"], d["v"], rel0, d["u"], d["v_bias"], M, L, 0.7)
    mask = torch.arange(M + L)[None, :] <= torch.arange(L)[:, None] + M
    qu = torch.from_numpy(d["q"] + d["u"][None, :, None, :])
    ref = torch.nn.functional.scaled_dot_product_attention(
        qu, torch.from_numpy(d["k"]), torch.from_numpy(d["v"]), attn_mask=mask, scale=0.7)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Brute force on tiny shapes (independent pure-Python implementation)
# ---------------------------------------------------------------------------

TINY = [(M, L, dh) for M, L, dh in itertools.product(range(4), range(1, 4), (1, 2, 4))]


@pytest.mark.parametrize("M,L,dh", TINY)
def test_brute_force_tiny(M, L, dh):
    B, H = 1, 2
    d = rand_heads(B, H, L, M, dh, seed=1000 + 16 * M + 4 * L + dh)
    scale = 0.9
    out, lse = oracle.relattn(d["q"], d["k"], d["v"], d["r"], d["u"], d["v_bias"], M, L, scale)
    for h in range(H):
        rel = d["r"][h]
        o_b, lse_b = brute.attention_from_tables(
            d["q"][0, h].tolist(), d["k"][0, h].tolist(), d["v"][0, h].tolist(),
            lambda dist, rel=rel: rel[dist].tolist(), d["u"][h].tolist(),
            d["v_bias"][h].tolist(), M, L, scale)
        np.testing.assert_allclose(out[0, h], np.array(o_b), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[0, h], np.array(lse_b), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("M,L,H", [(0, 3, 1), (2, 2, 2), (3, 1, 2)])
def test_brute_force_from_raw_states(M, L, H):
    # End-to-end from hidden states: projections, sinusoid table, W_kR R.
    dh, dmod = 2, 6
    g = torch.Generator().manual_seed(77 + M)
    h_ext = torch.randn(1, M + L, dmod, generator=g).double().numpy()
    W = [torch.randn(H * dh, dmod, generator=g).double().numpy() * 0.5 for _ in range(4)]
    u = torch.randn(H, dh, generator=g).double().numpy()
    vb = torch.randn(H, dh, generator=g).double().numpy()
    q, k, v, rel = oracle.attention_inputs(h_ext[:, M:], h_ext[:, :M], *W, H)
    out, _ = oracle.relattn(q, k, v, rel, u, vb, M, L, 0.8)
    ref = brute.layer_attention(h_ext.tolist(), *(w.tolist() for w in W), u.tolist(),
                                vb.tolist(), H, M, L, 0.8)
    np.testing.assert_allclose(out, np.array(ref), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# Shift invariance (§3.3: only relative distances enter the score)
# ---------------------------------------------------------------------------

def test_shift_of_absolute_positions_leaves_output_unchanged():
    M, L, H, dh, dmod = 3, 3, 1, 2, 4
    g = torch.Generator().manual_seed(5)
    h_ext = torch.randn(1, M + L, dmod, generator=g).double().numpy().tolist()
    W = [(torch.randn(H * dh, dmod, generator=g) * 0.5).double().numpy().tolist() for _ in range(4)]
    u = [[0.3, -0.2]]
    vb = [[-0.1, 0.4]]
    base = brute.layer_attention(h_ext, *W, u, vb, H, M, L, 1.0, offset=0)
    for c in (1, 17, 1000):
        moved = brute.layer_attention(h_ext, *W, u, vb, H, M, L, 1.0, offset=c)
        np.testing.assert_allclose(np.array(moved), np.array(base), rtol=1e-12, atol=1e-12)
    # Contrast (§3.3, A^abs): adding absolute encodings U_pos to the states is
    # not invariant to the same shift.
    def absolute(offset):
        hs = [[[x + y for x, y in zip(row, brute.sinusoid_row(offset + j, dmod))]
               for j, row in enumerate(h_ext[0])]]
        zero = lambda dist: [0.0] * dh
        Wq = W[0]
        q = [brute.matvec(Wq, hs[0][M + i]) for i in range(L)]
        k = [brute.matvec(W[1], x) for x in hs[0]]
        v = [brute.matvec(W[2], x) for x in hs[0]]
        return brute.attention_from_tables(q, k, v, zero, [0.0] * dh, [0.0] * dh, M, L, 1.0)[0]
    assert not np.allclose(absolute(0), absolute(17), atol=1e-6)


# ---------------------------------------------------------------------------
# Softmax invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,L", [(0, 4), (5, 6), (12, 3)])
def test_probabilities_sum_to_one_and_respect_mask(M, L):
    # With v = identity over the K keys the output rows are the softmax rows.
    K = M + L
    d = rand_heads(1, 1, L, M, 8, seed=400 + M)
    eye = np.eye(K)[None, None]
    # Keys and relative vectors keep width 8; v has width K.
    out, _ = _relattn_wide_v(d, eye, M, L)
    out = out[..., :K]
    np.testing.assert_allclose(out.sum(-1), 1.0, rtol=1e-13)
    ii, jj = np.meshgrid(np.arange(L), np.arange(K), indexing="ij")
    assert np.all(out[0, 0][jj > ii + M] == 0.0)
    assert np.all(out[0, 0][jj <= ii + M] > 0.0)


def _relattn_wide_v(d, v, M, L):
    # The C oracle takes one dh for all operands: pad q, k, r, u, v_bias with
    # zeros up to the width of v (zeros add nothing to the dot products).
    w = max(v.shape[-1], d["q"].shape[-1])
    pad = lambda x: np.concatenate([x, np.zeros(x.shape[:-1] + (w - x.shape[-1],))], axis=-1)
    return oracle.relattn(pad(d["q"]), pad(d["k"]), pad(v), pad(d["r"]), pad(d["u"]),
                          pad(d["v_bias"]), M, L, 0.5)


def test_output_in_convex_hull_of_visible_values():
    M, L = 6, 5
    d = rand_heads(1, 2, L, M, 4, seed=501)
    out, _ = oracle.relattn(d["q"], d["k"], d["v"], d["r"], d["u"], d["v_bias"], M, L, 0.5)
    for h in range(2):
        for i in range(L):
            vis = d["v"][0, h, : M + i + 1]
            assert np.all(out[0, h, i] <= vis.max(0) + 1e-12)
            assert np.all(out[0, h, i] >= vis.min(0) - 1e-12)


def test_bh_subset_matches_full():
    d = rand_heads(2, 3, 4, 5, 8, seed=601)
    full, lfull = oracle.relattn(d["q"], d["k"], d["v"], d["r"], d["u"], d["v_bias"], 5, 4, 0.4)
    part, lpart = oracle.relattn(d["q"], d["k"], d["v"], d["r"], d["u"], d["v_bias"], 5, 4, 0.4,
                                 bh=[4, 1])
    for bh in (4, 1):
        b, h = divmod(bh, 3)
        np.testing.assert_array_equal(part[b, h], full[b, h])
        np.testing.assert_array_equal(lpart[b, h], lfull[b, h])
    assert np.isnan(part[0, 0]).all()


# ---------------------------------------------------------------------------
# Layer glue of the stack model: LayerNorm and the position-wise feed-forward
# ---------------------------------------------------------------------------

def test_oracle_layer_glue():
    g = torch.Generator().manual_seed(71)
    B, L, d, hd, f = 2, 5, 12, 8, 20
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)
    a, h = r(B, L, hd), r(B, L, d)
    lay = {"W_o": r(d, hd), "b_o": r(d), "W_1": r(f, d), "b_1": r(f), "W_2": r(d, f), "b_2": r(d)}
    F = torch.nn.functional
    x = r(3, 7, d) * 3 + 1
    np.testing.assert_allclose(oracle.layer_norm(x.numpy()),
                               F.layer_norm(x, (d,), eps=oracle.LN_EPS).numpy(), rtol=1e-12,
                               atol=1e-12)
    o = F.layer_norm(F.linear(a, lay["W_o"], lay["b_o"]) + h, (d,), eps=1e-5)
    want = F.layer_norm(o + F.linear(F.relu(F.linear(o, lay["W_1"], lay["b_1"])), lay["W_2"],
                                     lay["b_2"]), (d,), eps=1e-5)
    got = oracle.layer_post(a.numpy(), h.numpy(), {k: v.numpy() for k, v in lay.items()})
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-11, atol=1e-11)
