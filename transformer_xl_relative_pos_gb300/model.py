"""Layer glue around the kernels: projections and the streaming N-layer stack.

"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
§3.3 N-layer summary, for n = 1..N:
    h~  = [SG(m^{n-1}) o h^{n-1}]                      -> mem_concat (kernel)
    q, k, v = h W_q^T, h~ W_kE^T, h~ W_v^T             -> torch matmul
    a   = Masked-Softmax(A) v                           -> relattn_fwd (kernel)
    o   = LayerNorm(Linear(a) + h^{n-1})                -> torch
    h^n = Positionwise-Feed-Forward(o)                  -> torch (ReLU MLP,
                                                           residual, LayerNorm)
and the memory of each layer advances to the newest M states of its input
(§3.2)                                                  -> mem_update (kernel).
With ``cache_kv`` the stack also keeps, per layer, rings of the memory's
projected keys and values: the memory rows and W_kE, W_v do not change at
evaluation, so k and v of the memory are the ones projected when those states
were the segment, and each segment projects only its own L rows (2·M·d²
multiply-adds saved per layer and projection); the rings are the same kernels
on a [B·H, M, d_head] view.  The attention takes k and v as one contiguous
tensor, so the rings are copied out every segment: replayed from CUDA graphs
the cached stack is slightly faster than re-projecting the memory (the saved
multiply-adds outweigh the copies), launched eagerly it is slower (four more
launches per layer), so it is off by default.
The relative table r = W_kR R is built from rel_pos_emb (kernel) and one matmul
and is cached per (layer, K): R has no parameters and W_kR is fixed at
evaluation.

With ``graphs`` the stack replays each segment from a CUDA graph once the
memories are full: every launch of a segment then has fixed shapes and
pointers, and the ring heads come back to the same positions every
M / gcd(M, L) segments, so one graph per ring position covers the stream (one
graph when L is a multiple of M).  The host-side ring states advance exactly
as the eager calls advance them.

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
        # projected memory: [B*H, M, dh] rings of k and v per layer, each with its
        # own ring state (they advance exactly as the hidden-state ring)
        ring = lambda: torch.zeros(B * self.H, self.M, self.dh, dtype=self.dtype, device=self.device)
        self.kmems = [ring() for _ in self.layers] if self.cache_kv else None
        self.vmems = [ring() for _ in self.layers] if self.cache_kv else None
        self.kv_states = ([(txl.MemState(0, 0, self.M), txl.MemState(0, 0, self.M))
                           for _ in self.layers] if self.cache_kv else None)

    def memories(self):
        """Each layer's memory in logical order (oldest first), [B, fill, d]."""
        out = []
        for mem, st in zip(self.mems, self.states):
            B = mem.shape[0]
            empty = torch.empty(B, 0, self.d, dtype=self.dtype, device=self.device)
            out.append(txl.mem_concat(mem, st, empty))
        return out

    def _r(self, n: int, K: int) -> torch.Tensor:
        key = (n, K)
        if key not in self._r_cache:
            R = txl.rel_pos_emb(K, self.d, dtype=torch.float32, device=self.device)
            self._r_cache[key] = rel_table_heads(R, self.layers[n]["W_kR"].float(),
                                                 self.H).to(self.dtype)
        return self._r_cache[key]

    def _rings(self):
        rings = list(self.states)
        if self.cache_kv:
            rings += [s for pair in self.kv_states for s in pair]
        return rings

    def segment(self, tokens: torch.Tensor) -> torch.Tensor:
        """One segment [B, L] -> the top layer's states [B, L, d].  With graphs
        the result lives in the graph's memory and is overwritten by the next
        replay of the same ring position."""
        B, L = tokens.shape
        if self.mems is None or self.mems[0].shape[0] != B:
            self.reset(B)
        full = self.M > 0 and self.states[0].fill == self.M
        # capture only after one eager segment at full memory (warm-up of the
        # library's and torch's lazily set-up state for these shapes)
        if not (self.graphs and full and self._full_segments >= 1):
            if full:
                self._full_segments += 1
            return self._segment(tokens.to(self.device))
        key = self.states[0].head
        if key not in self._graphs:
            saved = [(st.head, st.fill) for st in self._rings()]
            tok = torch.empty(B, L, dtype=torch.long, device=self.device)
            tok.copy_(tokens)
            graph = torch.cuda.CUDAGraph()
            if self._pool is None:
                self._pool = torch.cuda.graph_pool_handle()
            with torch.cuda.graph(graph, pool=self._pool):
                out = self._segment(tok)
            # capture recorded the launches without running them: put the ring
            # states back; the replay below runs the segment
            for st, (head, fill) in zip(self._rings(), saved):
                st.head, st.fill = head, fill
            self._graphs[key] = (graph, tok, out)
        graph, tok, out = self._graphs[key]
        tok.copy_(tokens)
        graph.replay()
        for st in self._rings():  # what the eager mem_update calls do on the host
            st.fill = min(st.fill + L, st.capacity)
            st.head = (st.head + L) % st.capacity
        return out

    def _segment(self, tokens: torch.Tensor) -> torch.Tensor:
        B, L = tokens.shape
        h = self.emb[tokens]
        for n, lay in enumerate(self.layers):
            st = self.states[n]
            M_cur = st.fill
            q = project_heads(h, lay["W_q"], self.H)
            if self.cache_kv:
                # only the segment's rows are projected; the memory's come from the rings
                ks, vs = self.kv_states[n]
                k_new = project_heads(h, lay["W_kE"], self.H).view(B * self.H, L, self.dh)
                v_new = project_heads(h, lay["W_v"], self.H).view(B * self.H, L, self.dh)
                k = txl.mem_concat(self.kmems[n], ks, k_new).view(B, self.H, M_cur + L, self.dh)
                v = txl.mem_concat(self.vmems[n], vs, v_new).view(B, self.H, M_cur + L, self.dh)
            else:
                ext = txl.mem_concat(self.mems[n], st, h)
                k = project_heads(ext, lay["W_kE"], self.H)
                v = project_heads(ext, lay["W_v"], self.H)
            r = self._r(n, M_cur + L)
            a_heads = txl.relattn_fwd(q, k, v, r, self.u, self.v_bias, M_cur, self.scale)
            a = a_heads.transpose(1, 2).reshape(B, L, -1)
            o = layer_norm((a @ lay["W_o"].t()).float() + lay["b_o"].float() + h.float())
            f = torch.relu(o.to(self.dtype) @ lay["W_1"].t() + lay["b_1"])
            h_next = layer_norm(o + (f @ lay["W_2"].t()).float() + lay["b_2"].float())
            if self.taps is not None:
                mem_now = txl.mem_concat(self.mems[n], st, h[:, :0])
                self.taps.append({"h": h, "mem": mem_now, "q": q, "k": k, "v": v, "r": r,
                                  "M": M_cur, "a": a_heads, "h_out": h_next.to(self.dtype)})
            txl.mem_update(self.mems[n], st, h)
            if self.cache_kv:
                txl.mem_update(self.kmems[n], ks, k_new)
                txl.mem_update(self.vmems[n], vs, v_new)
            h = h_next.to(self.dtype)
        return h
