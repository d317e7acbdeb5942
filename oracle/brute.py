"""Second, independently written brute force for tiny cases (pure Python).

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  It deliberately takes a
different route from the C oracle, so that the two pin each other:

  * positions are absolute: query i of the segment sits at position
    ``offset + M + i``, key j at ``offset + j``; the distance is their
    difference and a key is visible iff it is not after the query;
  * the score uses the compact grouping of §3.3 of "Transformer-XL: Attentive
    Language Models Beyond a Fixed-Length Context":
        A_ij = (q_i + u) . k_j + (q_i + v) . W_kR R_{i-j}
    instead of the four separate terms (a)-(d);
  * the sinusoid is written as sin(p / 10000^(2k/d)), cos(p / 10000^(2k/d)),
    and W_kR R_delta is formed from the raw weights for every pair.
"""

from __future__ import annotations

import math


def sinusoid_row(p: float, d: int):
    row = []
    for k in range(d // 2):
        denom = 10000.0 ** (2.0 * k / d)
        row.append(math.sin(p / denom))
        row.append(math.cos(p / denom))
    return row


def matvec(W, x):
    return [sum(W[a][c] * x[c] for c in range(len(x))) for a in range(len(W))]


def attention_from_tables(q, k, v, rel_fn, u, vb, M, L, scale, offset=0):
    """One head.  q [L][dh], k/v [M+L][dh] as nested lists; rel_fn(distance)
    returns the projected relative vector.  Returns (out [L][dh], lse [L])."""
    dh = len(v[0]) if v else 0
    out, lse = [], []
    for i in range(L):
        pos_q = offset + M + i
        qu = [q[i][t] + u[t] for t in range(len(u))]
        qv = [q[i][t] + vb[t] for t in range(len(vb))]
        logits = []
        for j in range(M + L):
            pos_k = offset + j
            if pos_k > pos_q:
                continue
            r = rel_fn(pos_q - pos_k)
            s = sum(qu[t] * k[j][t] for t in range(len(qu)))
            s += sum(qv[t] * r[t] for t in range(len(qv)))
            logits.append((j, scale * s))
        top = max(x for _, x in logits)
        weights = [(j, math.exp(x - top)) for j, x in logits]
        z = sum(w for _, w in weights)
        out.append([sum(w * v[j][t] for j, w in weights) / z for t in range(dh)])
        lse.append(top + math.log(z))
    return out, lse


def layer_attention(h_ext, W_q, W_kE, W_v, W_kR, u, vb, H, M, L, scale, offset=0):
    """Multi-head attention output a[b][h][i][t] from raw states.

    h_ext [B][M+L][d] (memory rows first), weights [H*dh][d], u/vb [H][dh]."""
    dh = len(W_q) // H
    d = len(h_ext[0][0])
    res = []
    for hb in h_ext:
        per_head = []
        for hh in range(H):
            rows = range(hh * dh, (hh + 1) * dh)
            Wq = [W_q[a] for a in rows]
            Wk = [W_kE[a] for a in rows]
            Wv = [W_v[a] for a in rows]
            Wr = [W_kR[a] for a in rows]
            q = [matvec(Wq, hb[M + i]) for i in range(L)]
            k = [matvec(Wk, x) for x in hb]
            v = [matvec(Wv, x) for x in hb]
            rel = lambda dist, Wr=Wr: matvec(Wr, sinusoid_row(dist, d))
            o, _ = attention_from_tables(q, k, v, rel, u[hh], vb[hh], M, L, scale, offset)
            per_head.append(o)
        res.append(per_head)
    return res
