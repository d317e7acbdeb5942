"""The streaming 12-layer stack on the GPU against the oracle's explicit
recomputation of the last segment from the stored memories.

"Transformer-XL: Attentive Language Models Beyond a Fixed-Length Context",
§3.2 (each layer caches the last M states of its input and reuses them as
extended context) and the §3.3 N-layer summary.  The GPU runs all segments
with its kernels (memory concat/update, positional table, attention) and torch
for projections, LayerNorm and the feed-forward.  Before the last segment its
memories are read back; the oracle then computes that segment in fp64 from
those memories with the same bf16-rounded parameters and the per-pair
relative vectors, and the top-layer states are compared.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import txl_inputs
from parity import TOL_BF16, TOL_BF16_RMS, compare, dev
import transformer_xl_relative_pos_gb300 as txl
from transformer_xl_relative_pos_gb300.model import XLStack

pytestmark = pytest.mark.gpu


def rounded(t, dtype=torch.bfloat16):
    return t.to(dtype).double().numpy()


def run_stack(w, n_layer=None, n_seg=None, cache_kv=False):
    params = txl_inputs.draw_stack(w)
    if n_layer is not None:
        params["layers"] = params["layers"][:n_layer]
    stack = XLStack(params, w.H, w.M, dev(), torch.bfloat16, cache_kv=cache_kv)
    tokens = params["tokens"][: (n_seg or w.n_seg)]
    for s in range(tokens.shape[0] - 1):
        stack.segment(tokens[s])
    mems = [m.double().cpu().numpy() for m in stack.memories()]
    h_gpu = stack.segment(tokens[-1]).double().cpu().numpy()
    torch.cuda.synchronize()
    layers64 = [{k: rounded(v) for k, v in lay.items()} for lay in params["layers"]]
    h_or, _ = oracle.segment_forward(tokens[-1].numpy(), rounded(params["emb"]), layers64, mems,
                                     rounded(params["u"]), rounded(params["v_bias"]), w.H, w.M,
                                     1.0 / math.sqrt(w.dh))
    return h_gpu, h_or, stack, mems


@pytest.mark.parametrize("cache_kv", [True, False])
def test_small_stack_memory_fill_and_wrap(cache_kv):
    # 3 layers, L=64 and M=100: the memories fill over two segments, then wrap.
    # With cache_kv the memory's keys and values come from the projected rings,
    # without it they are re-projected from the hidden-state memory.
    base = txl_inputs.WORKLOADS["c5_stack12_L512_M512"]
    w = txl_inputs.Workload("small_stack", B=2, H=2, dh=64, L=64, M=100, d_model=128,
                            dtype="bf16", seed=41, d_ff=256, n_layer=3, n_seg=5, vocab=base.vocab)
    h_gpu, h_or, stack, mems = run_stack(w, cache_kv=cache_kv)
    assert all(m.shape[1] == 100 for m in mems)
    # three layers: sqrt(3) times the one-layer bound (below) is 4.5e-2
    compare(h_gpu, h_or, 6e-2, 1.5e-2, what=f"small stack cache_kv={cache_kv}")


# Bounds of the stack checks.  The stack keeps its states in bf16 between layers
# (the workload's element type), so a layer's output carries up to half a bf16
# ulp of its magnitude: 2^-9 * 2^ceil(log2 max|h|), 0.0156 for the LayerNorm
# outputs here (|h| < 8).  Inside a layer the other bf16 rounding points (the
# attention output, the Linear outputs, o rounded for the feed-forward input)
# reach the output through weights ~N(0, 0.02) (a gain of about 0.02 * sqrt(fan-in)
# ~ 0.45 per matmul) and the LayerNorm's division by a standard deviation near 1:
# at most about 1e-2 on the largest outputs.  One layer: half an output ulp + 1e-2.
# Through N layers the residual stream carries each layer's error forward with a
# gain near 1 (LayerNorm of o + f, both O(1)); independent roundings add like a
# random walk, so N = 12 layers stay within 1e-1 at the maximum (sqrt(12) times
# the one-layer bound is 9e-2) and 2e-2 in rms (sqrt(12) times the one-layer rms
# bound is 1.7e-2).
LAYER_INTERNAL = 1e-2
LAYER_RMS = 5e-3


def half_ulp_bf16(x):
    m = float(np.abs(x).max())
    return 2.0 ** -9 * 2.0 ** math.ceil(math.log2(m)) if m > 0 else 0.0


@pytest.fixture(scope="module")
def c5_last_segment():
    """The 12-layer, 16-segment stream; the last segment runs with taps on every
    layer (input, memory, attention operands and output, layer output)."""
    w = txl_inputs.WORKLOADS["c5_stack12_L512_M512"]
    params = txl_inputs.draw_stack(w)
    stack = XLStack(params, w.H, w.M, dev(), torch.bfloat16)
    tokens = params["tokens"]
    for s in range(tokens.shape[0] - 1):
        stack.segment(tokens[s])
    mems = [m.double().cpu().numpy() for m in stack.memories()]
    stack.taps = []
    h_gpu = stack.segment(tokens[-1]).double().cpu().numpy()
    torch.cuda.synchronize()
    assert txl.device_status() == 0
    taps = [{k: (v.double().cpu().numpy() if torch.is_tensor(v) else v) for k, v in tp.items()}
            for tp in stack.taps]
    layers64 = [{k: rounded(v) for k, v in lay.items()} for lay in params["layers"]]
    return {"w": w, "params": params, "mems": mems, "h_gpu": h_gpu, "taps": taps,
            "layers64": layers64, "u": rounded(params["u"]), "v_bias": rounded(params["v_bias"])}


def test_c5_stack12_attention_of_every_layer(c5_last_segment):
    # Kernel parity inside the stream, at the stated tolerance: each layer's
    # attention output of the last segment against the fp64 oracle on that
    # layer's own bf16 q, k, v and table (§3.3 summary, one layer at a time).
    c = c5_last_segment
    w = c["w"]
    assert len(c["taps"]) == 12
    for n, tp in enumerate(c["taps"]):
        K = tp["k"].shape[2]
        assert tp["M"] == w.M and K == w.M + w.L
        rel = oracle.distance_table(tp["r"][:, -K:])
        want, _ = oracle.relattn(tp["q"], tp["k"], tp["v"], rel, c["u"], c["v_bias"], tp["M"],
                                 w.L, 1.0 / math.sqrt(w.dh))
        compare(tp["a"], want, TOL_BF16, TOL_BF16_RMS, what=f"c5 layer {n} attention")


def test_c5_stack12_every_layer_step(c5_last_segment):
    # Each layer of the last segment against the oracle's layer (§3.3 summary:
    # attention, Linear + residual + LayerNorm, feed-forward) run in fp64 on the
    # GPU layer's own bf16 input and memory; bound: half an output ulp plus the
    # propagated internal rounding (see the bounds above).
    c = c5_last_segment
    w = c["w"]
    for n, tp in enumerate(c["taps"]):
        want = oracle.layer_forward(tp["h"], tp["mem"], c["layers64"][n], c["u"], c["v_bias"],
                                    w.H, 1.0 / math.sqrt(w.dh))
        bound = half_ulp_bf16(want) + LAYER_INTERNAL
        err = np.abs(tp["h_out"] - want)
        assert float(err.max()) <= bound, f"layer {n}: max |err| {err.max():.3e} > {bound:.3e}"
        assert math.sqrt(float((err ** 2).mean())) <= LAYER_RMS, f"layer {n}: rms"
        if n + 1 < len(c["taps"]):  # the next layer reads exactly this output
            assert np.array_equal(c["taps"][n + 1]["h"], tp["h_out"])


def test_c5_stack12_last_segment(c5_last_segment):
    # The whole stream against the oracle's explicit recomputation of the last
    # segment from the stored memories (§3.2 recurrence, §3.3 summary); bound
    # from the one-layer bound compounded over 12 layers (see above).
    c = c5_last_segment
    w = c["w"]
    mems = c["mems"]
    assert len(mems) == 12 and all(m.shape == (w.B, w.M, w.d_model) for m in mems)
    h_or, _ = oracle.segment_forward(c["params"]["tokens"][-1].numpy(), rounded(c["params"]["emb"]),
                                     c["layers64"], mems, c["u"], c["v_bias"], w.H, w.M,
                                     1.0 / math.sqrt(w.dh))
    compare(c["h_gpu"], h_or, 1e-1, 2e-2, what="c5 top layer")


def test_cached_kv_windows_match_projected_memory():
    # After the memories have filled and the windows have moved back to their
    # buffers' front at least once, each layer's key and value windows hold the
    # projections of that layer's hidden-state memory.
    from transformer_xl_relative_pos_gb300.model import project_heads
    base = txl_inputs.WORKLOADS["c5_stack12_L512_M512"]
    w = txl_inputs.Workload("ring_stack", B=2, H=2, dh=64, L=48, M=100, d_model=128,
                            dtype="bf16", seed=43, d_ff=256, n_layer=3, n_seg=9, vocab=base.vocab)
    params = txl_inputs.draw_stack(w)
    stack = XLStack(params, w.H, w.M, dev(), torch.bfloat16, cache_kv=True)
    starts = set()
    for s in range(w.n_seg):
        stack.segment(params["tokens"][s])
        starts.add(stack.kv_windows[0].start)
    assert 0 in starts and len(starts) > 2
    for n, (mem, lay) in enumerate(zip(stack.memories(), stack.layers)):
        assert stack.kv_windows[n].fill == w.M
        k_win, v_win = stack.kv_memory(n)
        k_mem = project_heads(mem, lay["W_kE"], w.H)
        v_mem = project_heads(mem, lay["W_v"], w.H)
        # the same bf16 products, possibly summed in another order by the GEMM
        compare(k_win.float().cpu().numpy(), k_mem.float().cpu().numpy(), 5e-3, what=f"k window {n}")
        compare(v_win.float().cpu().numpy(), v_mem.float().cpu().numpy(), 5e-3, what=f"v window {n}")


@pytest.mark.parametrize("L,M,cache_kv", [(64, 64, False), (64, 128, True), (48, 80, False)])
def test_graph_replayed_stack_matches_eager(L, M, cache_kv):
    # Once the memories are full the stack replays each segment from a CUDA
    # graph per position of its rings (and windows); every segment's output and
    # the final memories must equal the eager stack's bit for bit (same
    # kernels, same order, same operands).
    base = txl_inputs.WORKLOADS["c5_stack12_L512_M512"]
    w = txl_inputs.Workload("graph_stack", B=2, H=2, dh=64, L=L, M=M, d_model=128,
                            dtype="bf16", seed=43, d_ff=256, n_layer=2, n_seg=10, vocab=base.vocab)
    params = txl_inputs.draw_stack(w)
    eager = XLStack(params, w.H, w.M, dev(), torch.bfloat16, cache_kv=cache_kv)
    graphed = XLStack(params, w.H, w.M, dev(), torch.bfloat16, cache_kv=cache_kv, graphs=True)
    for s in range(w.n_seg):
        want = eager.segment(params["tokens"][s]).clone()
        got = graphed.segment(params["tokens"][s]).clone()
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"segment {s}"
    # one graph per combination of ring heads and window starts: the ring heads
    # repeat every M / gcd(M, L) segments, the windows' starts (0, L, ..., C - M - L)
    # every (C - M - L) / L + 1, a multiple of that
    expected = M // math.gcd(M, L)
    if cache_kv:
        C = graphed.kv_windows[0].capacity
        expected = (C - M - L) // L + 1
        assert expected % (M // math.gcd(M, L)) == 0
    assert len(graphed._graphs) == expected
    for a, b in zip(eager.memories(), graphed.memories()):
        assert torch.equal(a, b)
    for sa, sb in zip(eager._host_states(), graphed._host_states()):
        assert XLStack._snap(sa) == XLStack._snap(sb)


@pytest.mark.parametrize("cache_kv,graphs", [(False, False), (True, False), (True, True)])
def test_checkpoint_resume_is_exact(cache_kv, graphs):
    # 16 segments straight against 8, a checkpoint to host memory, a fresh stack
    # restored from it, and 8 more: every output and the final memories equal the
    # straight run's bit for bit (§3.2: the memory is all the stream carries).
    base = txl_inputs.WORKLOADS["c5_stack12_L512_M512"]
    w = txl_inputs.Workload("ckpt_stack", B=2, H=2, dh=64, L=48, M=100, d_model=128,
                            dtype="bf16", seed=47, d_ff=256, n_layer=3, n_seg=16, vocab=base.vocab)
    params = txl_inputs.draw_stack(w)
    tokens = params["tokens"]
    straight = XLStack(params, w.H, w.M, dev(), torch.bfloat16, cache_kv=cache_kv, graphs=graphs)
    want = [straight.segment(tokens[s]).clone() for s in range(16)]
    first = XLStack(params, w.H, w.M, dev(), torch.bfloat16, cache_kv=cache_kv, graphs=graphs)
    for s in range(8):
        assert torch.equal(first.segment(tokens[s]), want[s])
    ck = first.checkpoint()
    assert all(not t.is_cuda for t in ck["mems"])
    del first
    second = XLStack(params, w.H, w.M, dev(), torch.bfloat16, cache_kv=cache_kv, graphs=graphs)
    second.restore(ck)
    for s in range(8, 16):
        got = second.segment(tokens[s]).clone()
        torch.cuda.synchronize()
        assert torch.equal(got, want[s]), f"segment {s}"
    for a, b in zip(straight.memories(), second.memories()):
        assert torch.equal(a, b)
    for sa, sb in zip(straight._host_states(), second._host_states()):
        assert XLStack._snap(sa) == XLStack._snap(sb)
