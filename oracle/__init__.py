"""fp64 CPU oracle for Transformer-XL relative-position attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``transformer_xl_relative_pos_gb300``) and neither
imports the other; the seeded draws in ``txl_inputs`` feed both.

Source: "Transformer-XL: Attentive Language Models Beyond a Fixed-Length
Context" (Dai et al.):
  * §3.3, the four-term relative score A^rel (terms (a)-(d));
  * §3.3, the N-layer computational summary (extended context [SG(m) o h],
    masked softmax, Linear + residual + LayerNorm, position-wise feed-forward);
  * §3.2, the memory of the last M hidden states per layer, and training
    that backpropagates within a segment (``relattn_bwd``: the chain rule of
    the forward above, the memory SG(m));
  * Appendix B, the reversed table Q and the left-shift relation between
    B~ = q Q^T and B (used here only as a self-check, never for the result).

The per-pair attention loops are plain C (``txl_oracle.c``), compiled with gcc
and loaded through ctypes; everything else is numpy in fp64.  Every pin that
ties this oracle to the pages lives in ``tests/test_oracle_*.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "txl_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_txl.so")
_lock = threading.Lock()
_lib = None

LN_EPS = 1e-5  # LayerNorm epsilon (the pages give none; the common default)


def build(force: bool = False) -> str:
    """Compile ``txl_oracle.c`` into ``liboracle_txl.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # The mutation test points this at a deliberately broken build.
            override = os.environ.get("TXL_ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            lib.txlo_sinusoid_table.argtypes = [dp, ctypes.c_int, ctypes.c_int]
            lib.txlo_sinusoid_table.restype = ctypes.c_int
            lib.txlo_score_terms.argtypes = [dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, dp, dp, dp, dp, ip]
            lib.txlo_score_terms.restype = ctypes.c_int
            lib.txlo_relattn.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_double, ip, ctypes.c_int, ctypes.c_int]
            lib.txlo_relattn.restype = ctypes.c_int
            lib.txlo_relattn_bwd.argtypes = [dp] * 13 + [ctypes.c_int] * 5 + [ctypes.c_double,
                                                                                 ctypes.c_int]
            lib.txlo_relattn_bwd.restype = ctypes.c_int
            lib.txlo_max_threads.argtypes = []
            lib.txlo_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().txlo_max_threads())


# ----------------------------------------------------------------------------
# Positional table (§3.3: R is the sinusoid encoding matrix, row p = distance p)
# ----------------------------------------------------------------------------

def sinusoid_table(n_dist: int, d: int) -> np.ndarray:
    """R[p, :] for p in [0, n_dist): R_p[2k] = sin(p w_k), R_p[2k+1] = cos(p w_k),
    w_k = 10000^(-2k/d)."""
    R = np.empty((n_dist, d), dtype=np.float64)
    if _load().txlo_sinusoid_table(_dp(R), int(n_dist), int(d)) != 0:
        raise ValueError("sinusoid_table: need n_dist >= 0 and an even d > 0")
    return R


def reversed_table(rel_by_distance: np.ndarray) -> np.ndarray:
    """Appendix B's Q: row k holds W_kR R_{M+L-1-k}, i.e. the distance table in
    reversed row order.  Works on [..., K, dh] arrays."""
    return np.ascontiguousarray(np.flip(_f64(rel_by_distance), axis=-2))


def distance_table(reversed_rows: np.ndarray) -> np.ndarray:
    """Inverse of :func:`reversed_table`."""
    return np.ascontiguousarray(np.flip(_f64(reversed_rows), axis=-2))


# ----------------------------------------------------------------------------
# Attention (§3.3 A^rel, masked softmax, times v)
# ----------------------------------------------------------------------------

def relattn(q, k, v, rel, u, v_bias, M: int, L: int, scale: float,
            bh=None, nthreads: int = 0):
    """Relative-position attention over the extended context.

    q [B,H,L,dh]; k, v [B,H,M+L,dh] (memory rows first); rel [H,M+L,dh] with
    rel[h, delta] = W_kR,h R_delta (by distance); u, v_bias [H,dh].
    Returns (out [B,H,L,dh], lse [B,H,L]) in fp64 (lse in natural log).
    ``bh`` optionally lists flattened b*H+h pairs to compute; the others are NaN.
    """
    q, k, v, rel, u, v_bias = (_f64(t) for t in (q, k, v, rel, u, v_bias))
    B, H, Lq, dh = q.shape
    K = M + L
    if Lq != L or k.shape != (B, H, K, dh) or v.shape != (B, H, K, dh):
        raise ValueError("relattn: shape mismatch")
    if rel.shape != (H, K, dh) or u.shape != (H, dh) or v_bias.shape != (H, dh):
        raise ValueError("relattn: rel/u/v_bias shape mismatch")
    out = np.full((B, H, L, dh), np.nan)
    lse = np.full((B, H, L), np.nan)
    if bh is None:
        lst, n = None, B * H
    else:
        arr = np.ascontiguousarray(np.asarray(bh, dtype=np.int32))
        lst, n = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), int(arr.size)
    rc = _load().txlo_relattn(_dp(q), _dp(k), _dp(v), _dp(rel), _dp(u), _dp(v_bias),
                              _dp(out), _dp(lse), B, H, int(M), int(L), dh, float(scale),
                              lst, n, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"txlo_relattn failed ({rc})")
    return out, lse


def relattn_bwd(q, k, v, rel, u, v_bias, dout, M: int, L: int, scale: float,
                nthreads: int = 0):
    """Gradients of :func:`relattn`'s output against ``dout`` (training within a
    segment, §3.2; the memory rows are SG(m), yet their projected k and v get
    gradients like the segment's).

    Shapes as :func:`relattn`; dout [B,H,L,dh].  Returns fp64
    (dq [B,H,L,dh], dk [B,H,M+L,dh], dv [B,H,M+L,dh], drel [H,M+L,dh] by
    distance, du [H,dh], dvb [H,dh]); drel, du, dvb are summed over the batch.
    """
    q, k, v, rel, u, v_bias, dout = (_f64(t) for t in (q, k, v, rel, u, v_bias, dout))
    B, H, Lq, dh = q.shape
    K = M + L
    if Lq != L or k.shape != (B, H, K, dh) or v.shape != (B, H, K, dh) or dout.shape != q.shape:
        raise ValueError("relattn_bwd: shape mismatch")
    if rel.shape != (H, K, dh) or u.shape != (H, dh) or v_bias.shape != (H, dh):
        raise ValueError("relattn_bwd: rel/u/v_bias shape mismatch")
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    drel, du, dvb = np.empty_like(rel), np.empty_like(u), np.empty_like(v_bias)
    rc = _load().txlo_relattn_bwd(_dp(q), _dp(k), _dp(v), _dp(rel), _dp(u), _dp(v_bias),
                                  _dp(dout), _dp(dq), _dp(dk), _dp(dv), _dp(drel), _dp(du),
                                  _dp(dvb), B, H, int(M), int(L), dh, float(scale),
                                  int(nthreads))
    if rc != 0:
        raise RuntimeError(f"txlo_relattn_bwd failed ({rc})")
    return dq, dk, dv, drel, du, dvb


def score_terms(q, k, rel, u, v_bias, M: int, L: int):
    """The four unscaled terms (a), (b), (c), (d) of one head as [L, M+L]
    arrays, plus the validity mask (key j at or before query i)."""
    q, k, rel, u, v_bias = (_f64(t) for t in (q, k, rel, u, v_bias))
    K = M + L
    dh = q.shape[-1]
    ta, tb, tc, td = (np.empty((L, K)) for _ in range(4))
    valid = np.empty((L, K), dtype=np.int32)
    rc = _load().txlo_score_terms(_dp(q), _dp(k), _dp(rel), _dp(u), _dp(v_bias),
                                  int(M), int(L), int(dh), _dp(ta), _dp(tb), _dp(tc),
                                  _dp(td), valid.ctypes.data_as(ctypes.POINTER(ctypes.c_int)))
    if rc != 0:
        raise RuntimeError("txlo_score_terms failed")
    return ta, tb, tc, td, valid.astype(bool)


def appendix_b_position_term(q, rel, M: int, L: int):
    """Appendix B's linear-cost route to term (b): B~ = q Q^T with the reversed
    table Q, then row i of B is row i of B~ shifted left by L-1-i (entries that
    fall off the right end are the masked zeros).  Self-check only."""
    q, rel = _f64(q), _f64(rel)
    K = M + L
    Qrev = reversed_table(rel)          # Q_k = W_kR R_{M+L-1-k}
    Bt = q @ Qrev.T                     # [L, K]
    Bm = np.zeros((L, K))
    for i in range(L):
        s = L - 1 - i
        Bm[i, : K - s] = Bt[i, s:]
    return Bm


# ----------------------------------------------------------------------------
# Layer, stack and memory (§3.3 N-layer summary, §3.2 memory of length M)
# ----------------------------------------------------------------------------

def layer_norm(x: np.ndarray) -> np.ndarray:
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + LN_EPS)


def project_heads(x: np.ndarray, W: np.ndarray, H: int) -> np.ndarray:
    """x [B, T, d] times W^T ([H*dh, d]) -> [B, H, T, dh]."""
    B, T, _ = x.shape
    y = x @ W.T
    return np.ascontiguousarray(y.reshape(B, T, H, -1).transpose(0, 2, 1, 3))


def attention_inputs(h, mem, W_q, W_kE, W_v, W_kR, H: int):
    """q, k, v and the by-distance relative table of one layer.

    h [B, L, d] current segment, mem [B, M, d] (M may be 0).  The extended
    context is [SG(mem) o h] along the length; SG is the identity in a forward
    pass.  rel[h, delta] = W_kR,h R_delta for delta in [0, M+L)."""
    h, mem = _f64(h), _f64(mem)
    W_q, W_kE, W_v, W_kR = (_f64(w) for w in (W_q, W_kE, W_v, W_kR))
    ext = np.concatenate([mem, h], axis=1)
    K, d = ext.shape[1], ext.shape[2]
    q = project_heads(h, W_q, H)
    k = project_heads(ext, W_kE, H)
    v = project_heads(ext, W_v, H)
    R = sinusoid_table(K, d)
    rel = np.ascontiguousarray((R @ W_kR.T).reshape(K, H, -1).transpose(1, 0, 2))
    return q, k, v, rel


def layer_forward(h, mem, lay: dict, u, v_bias, H: int, scale: float, bh=None):
    """One Transformer-XL layer (§3.3 summary) on segment h with memory mem.

    a = Masked-Softmax(A) v;  o = LayerNorm(Linear(a) + h);
    h' = LayerNorm(o + W_2 ReLU(W_1 o + b_1) + b_2)."""
    h, mem = _f64(h), _f64(mem)
    M, L = mem.shape[1], h.shape[1]
    q, k, v, rel = attention_inputs(h, mem, lay["W_q"], lay["W_kE"], lay["W_v"],
                                    lay["W_kR"], H)
    a, _ = relattn(q, k, v, rel, u, v_bias, M, L, scale)
    B = h.shape[0]
    a = a.transpose(0, 2, 1, 3).reshape(B, L, -1)
    return layer_post(a, h, lay)


def layer_post(a, h, lay: dict):
    """The rest of the layer after attention (§3.3 summary):
    o = LayerNorm(Linear(a) + h);  h' = LayerNorm(o + W_2 ReLU(W_1 o + b_1) + b_2)."""
    a, h = _f64(a), _f64(h)
    o = layer_norm(a @ _f64(lay["W_o"]).T + _f64(lay["b_o"]) + h)
    f = np.maximum(o @ _f64(lay["W_1"]).T + _f64(lay["b_1"]), 0.0)
    return layer_norm(o + f @ _f64(lay["W_2"]).T + _f64(lay["b_2"]))


def memory_update(mem: np.ndarray, h: np.ndarray, M: int) -> np.ndarray:
    """§3.2: the memory caches the last M hidden states, oldest first:
    the newest M rows of [mem o h]."""
    ext = np.concatenate([_f64(mem), _f64(h)], axis=1)
    return np.ascontiguousarray(ext[:, max(0, ext.shape[1] - M):, :])


def segment_forward(tokens, emb, layers, mems, u, v_bias, H: int, M: int, scale: float):
    """One segment through the N-layer stack with per-layer memories.

    mems[n] holds the cached inputs of layer n (h^{n} in the pages' 1-based
    notation is the input of layer n+1; h^0 is the word embedding).  Returns the
    top-layer output and the advanced memories."""
    h = _f64(emb)[np.asarray(tokens)]
    new_mems = []
    for n, lay in enumerate(layers):
        new_mems.append(memory_update(mems[n], h, M))
        h = layer_forward(h, mems[n], lay, u, v_bias, H, scale)
    return h, new_mems


def empty_memories(n_layer: int, B: int, d: int):
    return [np.zeros((B, 0, d)) for _ in range(n_layer)]
