"""Layer glue around the kernels: projections and the streaming N-layer stack.

"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
§3.3 N-layer summary, for n = 1..N:
    h~  = [SG(m^{n-1}) o h^{n-1}]                      -> mem_concat (kernel)
    q, k, v = h W_q^T, h~ W_kE^T, h~ W_v^T             -> torch matmul (one
                                                           GEMM per operand set)
    a   = Masked-Softmax(A) v                           -> relattn_fwd (kernel)
    o   = LayerNorm(Linear(a) + h^{n-1})                -> torch
    h^n = Positionwise-Feed-Forward(o)                  -> torch (ReLU MLP,
                                                           residual, LayerNorm)
and the memory of each layer advances to the newest M states of its input
(§3.2)                                                  -> mem_update (kernel).
With ``cache_kv`` the stack also keeps, per layer, the memory's projected keys
and values: the memory rows and W_kE, W_v do not change at evaluation, so k and
v of the memory are the ones projected when those states were the segment, and
each segment projects only its own L rows (2·M·d² multiply-adds saved per layer
and projection).  Keys and values of a layer live in one window of a buffer
[2·B·H, capacity, d_head] (the keys' planes, then the values'): one launch of
txl_qkv_project computes the segment's q, k and v (one GEMM over the stacked
weights), writes k and v behind the memory's rows in the window and advances the
hidden-state memory ring; the attention reads [memory ; segment] in place, with
no copy of the memory per segment (txl_kv_window_advance after it).
The relative table r = W_kR R is built from rel_pos_emb (kernel) and one matmul
and is cached per (layer, K): R has no parameters and W_kR is fixed at
evaluation.

With ``graphs`` the stack replays each segment from a CUDA graph once the
memories are full: every launch of a segment then has fixed shapes and
pointers, and the ring heads and window starts come back to the same positions
periodically (every M / gcd(M, L) segments for the rings), so one graph per
combination of positions covers the stream.  A capture records the states the
eager calls leave behind, and a replay sets the host-side states to them.

Torch is used here for the dense projections, LayerNorm and the feed-forward
only; the attention, the positional table and the memory run in the CUDA
library.
"""

from __future__ import annotations

import math

import torch

from . import _lib as txl

LN_EPS = 1e-5


def project_heads(x: torch.Tensor, W: torch.Tensor, H: int) -> torch.Tensor:
    """x [B, T, d] times W^T ([H*dh, d]) -> contiguous [B, H, T, dh]."""
    B, T, _ = x.shape
    y = x @ W.t()
    return y.view(B, T, H, -1).transpose(1, 2).contiguous()


def project_stacked(x: torch.Tensor, W: torch.Tensor, n: int, H: int) -> torch.Tensor:
    """x [B, T, d] times W^T for W = [W_1; ...; W_n] (each [H*dh, d]) in one
    GEMM -> contiguous [n, B, H, T, dh] (operand i at index i)."""
    B, T, _ = x.shape
    y = x @ W.t()
    return y.view(B, T, n, H, -1).permute(2, 0, 3, 1, 4).contiguous()


def rel_table_heads(R_rev: torch.Tensor, W_kR: torch.Tensor, H: int) -> torch.Tensor:
    """r = R W_kR^T split per head: [K, d] x [H*dh, d]^T -> [H, K, dh]."""
    K = R_rev.shape[0]
    return (R_rev @ W_kR.t()).view(K, H, -1).transpose(0, 1).contiguous()


def attention_operands(h_ext, M: int, W_q, W_kE, W_v, W_kR, R_rev, H: int, dtype):
    """q, k, v, r for one layer from the extended context h_ext [B, M+L, d]
    (memory rows first) and the reversed table R_rev [M+L, d].  Products are
    formed in fp32 and rounded once to ``dtype``."""
    f = lambda t: t.float()
    h = f(h_ext)
    q = project_heads(h[:, M:], f(W_q), H).to(dtype)
    k = project_heads(h, f(W_kE), H).to(dtype)
    v = project_heads(h, f(W_v), H).to(dtype)
    r = rel_table_heads(f(R_rev), f(W_kR), H).to(dtype)
    return q, k, v, r


def layer_norm(x: torch.Tensor) -> torch.Tensor:
    return torch.nn.functional.layer_norm(x.float(), (x.shape[-1],), eps=LN_EPS)


class XLStack:
    """Evaluation-mode Transformer-XL stack with per-layer ring-buffer memories.

    params: draws from ``txl_inputs.draw_stack`` (CPU fp32); weights are moved
    to ``device`` in ``dtype``.  ``segment(tokens)`` processes one segment
    [B, L] and returns the top layer's states [B, L, d] (``dtype``)."""

    def __init__(self, params: dict, H: int, M: int, device, dtype=torch.bfloat16,
                 cache_kv: bool = False, graphs: bool = False):
        self.H, self.M, self.dtype, self.device = H, M, dtype, torch.device(device)
        self.cache_kv = cache_kv
        self.graphs = graphs
        self._graphs = {}        # ring head -> (graph, token buffer, output)
        self._pool = None
        self._full_segments = 0  # eager segments run with full memories
        to = lambda t: t.to(device=self.device, dtype=dtype).contiguous()
        self.emb = to(params["emb"])
        self.u = to(params["u"])
        self.v_bias = to(params["v_bias"])
        self.layers = [{k: to(v) for k, v in lay.items()} for lay in params["layers"]]
        for lay in self.layers:
            # stacked projection weights: q, k, v of the segment (cached k/v) or
            # k, v of the extended context (re-projection) in one GEMM
            lay["W_qkv"] = torch.cat([lay["W_q"], lay["W_kE"], lay["W_v"]]).contiguous()
            lay["W_kv"] = torch.cat([lay["W_kE"], lay["W_v"]]).contiguous()
        self.d = self.emb.shape[1]
        self.dh = self.u.shape[1]
        self.scale = 1.0 / math.sqrt(self.dh)
        self.mems = None
        self.states = None
        self._r_cache = {}
        # When set to a list, each eager segment appends, per layer, the layer's
        # input h, its memory, the attention operands (q, k, v, r, M), the
        # attention output a [B, H, L, dh] and the layer's output h' (all on the
        # device): what a per-layer check of the stack needs.
        self.taps = None

    def reset(self, B: int):
        self._graphs = {}
        self._full_segments = 0
        self.mems = [torch.zeros(B, self.M, self.d, dtype=self.dtype, device=self.device)
                     for _ in self.layers]
        self.states = [txl.MemState(0, 0, self.M) for _ in self.layers]
        # projected memory: k and v of each layer in one window of a
        # [2*B*H, C, dh] buffer; capacity C = M + n*L with n the smallest
        # multiple of the ring period M / gcd(M, L) that keeps C >= 2M + L
        # (window positions then repeat with the rings')
        self.kvbufs = self.kv_windows = None
        self._kv_L = None

    def _kv_reset(self, B: int, L: int):
        period = self.M // math.gcd(self.M, L) if self.M > 0 else 1
        n = period * max(1, -(-(self.M + L) // (period * L)))
        C = self.M + n * L
        self.kvbufs = [torch.zeros(2 * B * self.H, C, self.dh, dtype=self.dtype, device=self.device)
                       for _ in self.layers]
        self.kv_windows = [txl.KVWindow(0, 0, C, self.M) for _ in self.layers]
        self._kv_L = L
        self._graphs = {}
        self._full_segments = 0

    def checkpoint(self) -> dict:
        """Host copy of everything the stream carries from one segment to the
        next (§3.2: the memory of each layer; with cache_kv also the windows of
        projected keys and values), with the host-side ring and window states.
        ``restore`` on a fresh stack continues the stream exactly."""
        if self.mems is None:
            raise RuntimeError("checkpoint: no segment has run yet")
        torch.cuda.synchronize(self.device)
        ck = {"mems": [m.cpu() for m in self.mems],
              "states": [self._snap(st) for st in self.states], "kv": None}
        if self.cache_kv and self.kvbufs is not None:
            ck["kv"] = {"L": self._kv_L, "bufs": [b.cpu() for b in self.kvbufs],
                        "windows": [self._snap(w) for w in self.kv_windows]}
        return ck

    def restore(self, ck: dict):
        """Load a ``checkpoint`` (same parameters, shapes and options)."""
        B = ck["mems"][0].shape[0]
        self.reset(B)
        for mem, saved, st, snap in zip(self.mems, ck["mems"], self.states, ck["states"]):
            mem.copy_(saved)
            self._restore(st, snap)
        if ck["kv"] is not None:
            if not self.cache_kv:
                raise ValueError("restore: the checkpoint holds key/value windows")
            self._kv_reset(B, ck["kv"]["L"])
            for buf, saved in zip(self.kvbufs, ck["kv"]["bufs"]):
                buf.copy_(saved)
            for w, snap in zip(self.kv_windows, ck["kv"]["windows"]):
                self._restore(w, snap)
        torch.cuda.synchronize(self.device)

    def memories(self):
        """Each layer's memory in logical order (oldest first), [B, fill, d]."""
        out = []
        for mem, st in zip(self.mems, self.states):
            B = mem.shape[0]
            empty = torch.empty(B, 0, self.d, dtype=self.dtype, device=self.device)
            out.append(txl.mem_concat(mem, st, empty))
        return out

    def kv_memory(self, n: int):
        """Layer n's cached projected memory (cache_kv): keys and values
        [B, H, fill, dh], views into its window buffer."""
        w = self.kv_windows[n]
        kv = self.kvbufs[n][:, w.start:w.start + w.fill]
        kv = kv.view(2, -1, self.H, w.fill, self.dh)
        return kv[0], kv[1]

    def _r(self, n: int, K: int) -> torch.Tensor:
        key = (n, K)
        if key not in self._r_cache:
            R = txl.rel_pos_emb(K, self.d, dtype=torch.float32, device=self.device)
            self._r_cache[key] = rel_table_heads(R, self.layers[n]["W_kR"].float(),
                                                 self.H).to(self.dtype)
        return self._r_cache[key]

    def _host_states(self):
        """Every host-side memory state a segment advances (rings, windows)."""
        sts = list(self.states)
        if self.cache_kv and self.kv_windows is not None:
            sts += self.kv_windows
        return sts

    @staticmethod
    def _snap(st):
        return tuple(getattr(st, f) for f, _ in st._fields_)

    @staticmethod
    def _restore(st, snap):
        for (f, _), v in zip(st._fields_, snap):
            setattr(st, f, v)

    def segment(self, tokens: torch.Tensor) -> torch.Tensor:
        """One segment [B, L] -> the top layer's states [B, L, d].  With graphs
        the result lives in the graph's memory and is overwritten by the next
        replay of the same ring position."""
        B, L = tokens.shape
        if self.mems is None or self.mems[0].shape[0] != B:
            self.reset(B)
        if self.cache_kv and (self.kvbufs is None or self._kv_L != L):
            self._kv_reset(B, L)
        full = self.M > 0 and self.states[0].fill == self.M
        # capture only after one eager segment at full memory (warm-up of the
        # library's and torch's lazily set-up state for these shapes)
        if not (self.graphs and full and self._full_segments >= 1):
            if full:
                self._full_segments += 1
            return self._segment(tokens.to(self.device))
        sts = self._host_states()
        key = tuple(self._snap(st) for st in sts)
        if key not in self._graphs:
            tok = torch.empty(B, L, dtype=torch.long, device=self.device)
            tok.copy_(tokens)
            graph = torch.cuda.CUDAGraph()
            if self._pool is None:
                self._pool = torch.cuda.graph_pool_handle()
            with torch.cuda.graph(graph, pool=self._pool):
                out = self._segment(tok)
            # capture recorded the launches without running them: keep the
            # states the calls left behind for every replay, put the current
            # ones back; the replay below runs the segment
            after = [self._snap(st) for st in sts]
            for st, snap in zip(sts, key):
                self._restore(st, snap)
            self._graphs[key] = (graph, tok, out, after)
        graph, tok, out, after = self._graphs[key]
        tok.copy_(tokens)
        graph.replay()
        for st, snap in zip(sts, after):
            self._restore(st, snap)
        return out

    def _segment(self, tokens: torch.Tensor) -> torch.Tensor:
        B, L = tokens.shape
        h = self.emb[tokens]
        for n, lay in enumerate(self.layers):
            st = self.states[n]
            M_cur = st.fill
            mem_now = None
            if self.taps is not None:  # the memory this layer attends to
                mem_now = txl.mem_concat(self.mems[n], st, h[:, :0])
            if self.cache_kv:
                # only the segment's rows are projected: one launch computes q,
                # k, v (one GEMM over the stacked weights), writes k and v behind
                # the memory's rows in the window and advances the memory ring;
                # the attention reads [memory ; segment] in place
                kw = self.kv_windows[n]
                q = torch.empty(B, self.H, L, self.dh, dtype=self.dtype, device=self.device)
                txl.qkv_project(h, lay["W_qkv"], self.kvbufs[n], kw, q=q, mem=self.mems[n],
                                mem_state=st)
                kv = txl.kv_window_view(self.kvbufs[n], kw, L, 2 * B, self.H)
                kv = kv.view(2, B, self.H, -1, self.dh)
                k, v = kv[0], kv[1]
            else:
                q = project_heads(h, lay["W_q"], self.H)
                ext = txl.mem_concat(self.mems[n], st, h)
                kv = project_stacked(ext, lay["W_kv"], 2, self.H)
                k, v = kv[0], kv[1]
            r = self._r(n, M_cur + L)
            a_heads = txl.relattn_fwd(q, k, v, r, self.u, self.v_bias, M_cur, self.scale)
            a = a_heads.transpose(1, 2).reshape(B, L, -1)
            o = layer_norm((a @ lay["W_o"].t()).float() + lay["b_o"].float() + h.float())
            f = torch.relu(o.to(self.dtype) @ lay["W_1"].t() + lay["b_1"])
            h_next = layer_norm(o + (f @ lay["W_2"].t()).float() + lay["b_2"].float())
            if self.taps is not None:
                self.taps.append({"h": h, "mem": mem_now, "q": q, "k": k, "v": v, "r": r,
                                  "M": M_cur, "a": a_heads, "h_out": h_next.to(self.dtype)})
            if self.cache_kv:
                txl.kv_window_advance(kw, L)  # (the ring advanced in qkv_project)
            else:
                txl.mem_update(self.mems[n], st, h)
            h = h_next.to(self.dtype)
        return h
