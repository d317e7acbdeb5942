#!/usr/bin/env python3
"""Benchmark of the Transformer-XL relative-attention hot path on GB300.

A step is one layer-segment of evaluation with state reuse ("Transformer-XL:
Attentive Language Models Beyond a Fixed-Length Context", §3.2 and §3.3), at
the word-level large evaluation shape: batch 16, 16 heads of 64, segment
L = 128, memory M = 1600 (K = 1728 keys), d_model = 1024, bf16 operands:
    txl_relattn_fwd   fused relative-position attention (tcgen05/TMEM/TMA)
    txl_mem_update    memory ring advanced by the segment's L states
The q/k/v projections (torch matmuls) are set-up work outside the step, as the
attention operands of an evaluation segment.  The sinusoid table R
(txl_rel_pos_emb) and its projection r = W_kR R depend only on the layer and
the key count, so an evaluation computes them once per layer and reuses them
for every segment: they are built before the step, and the table kernel's own
time is reported beside the line (``rel_pos_emb_us``).

Metric: relative-attention forward TFLOP/s (6*L*K*d_head FLOPs per head and
call, masked entries included) plus tokens/s and the fraction of the measured
bf16 tensor-core peak.

Timing: W eager warm-up steps, then K steps replayed from a CUDA graph (the
graph holds the same launches; it removes host launch overhead), bracketed by
a barrier and device synchronisation, timed with CUDA events on the launching
stream, max over ranks.  Three input sets rotate so that every step's inputs
were last touched more than two L2-sizes of traffic ago.  The timed graph holds
no events of its own (an event recorded inside a graph costs several
microseconds of the step); the attention kernel's launch time comes from a
graph of back-to-back attention launches on the same input sets, timed right
after the timed region.

End to end (the line's ``e2e``): the recurrent evaluation through the public
API from pinned host buffers: each step copies in the new segment's q, k, v
and hidden states, appends k and v behind the device-resident memory windows
(txl_kv_window_append), attends over all K keys read in place from those
windows (txl_relattn_fwd_strided), advances the windows and the hidden-state
ring (txl_mem_update) and reads the output back; host clock around the steps.

``--impl reference`` times the fp64 CPU oracle instead (the reference arm).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import txl_inputs  # noqa: E402

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one attention
# launch on the headline workload, from one ncu --set full capture of this
# bench.  It is reported only while the kernel's sources are byte-identical to
# the ones that were profiled (else null).
PROFILED_TRAFFIC = {
    "workload": "c3_word_large_L128_M1600",
    "sources": ("relattn_tc.cu", "ptx.cuh", "kernels.h"),
    "sha256": "10af1cd26231feb98175aa8b69ea255436175eeed89233452dbd7c85e0294582",
    "bytes_per_launch": 121095424 + 2810880,
}


def profiled_traffic(workload_name: str):
    """DRAM bytes per attention launch if the profiled kernel is the one built, else None."""
    if workload_name != PROFILED_TRAFFIC["workload"]:
        return None
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "transformer_xl_relative_pos_gb300", "csrc")
    h = hashlib.sha256()
    for name in PROFILED_TRAFFIC["sources"]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return PROFILED_TRAFFIC["bytes_per_launch"] if h.hexdigest() == PROFILED_TRAFFIC["sha256"] else None


METRIC = "rel-attn fwd TFLOP/s + tokens/s at L=128,M=1600; % of GB300 bf16 TC peak"
N_SETS = 3
GRAPH_CHUNK = 1500      # steps per graph when K is large (multiple of 3 * 25)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stack", action="store_true",
                    help="per-segment time of the 12-layer streaming stack (config 5), with and "
                         "without cached projected memory keys/values, instead of the headline step")
    ap.add_argument("--table9", action="store_true",
                    help="per-token evaluation time, vanilla window recompute vs state reuse "
                         "(one attention layer), instead of the headline step")
    ap.add_argument("--decode", action="store_true",
                    help="time decode-shaped calls (a few new tokens against a long memory) "
                         "and their HBM bandwidth, instead of the headline step")
    ap.add_argument("--configs", action="store_true",
                    help="time one attention call of every bf16 workload shape, instead of the "
                         "headline step")
    ap.add_argument("--shapes", nargs="*", default=None,
                    help="with --decode: B,L,M triples (default: the long-memory decode set)")
    ap.add_argument("--calls", type=int, default=10,
                    help="with --decode or --configs: graph replays timed per shape (30 calls each)")
    ap.add_argument("--project", action="store_true",
                    help="time one layer's fused projection (txl_qkv_project) at the 12-layer "
                         "stream's shape against the unfused calls it replaces")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward (txl_relattn_bwd) at the headline shape (or the first "
                         "--workload), instead of the headline step")
    ap.add_argument("--workload", nargs="*", default=None,
                    help="with --configs: only these workloads; with --bwd: the workload to time "
                         "(names as in txl_inputs.WORKLOADS, bf16 ones)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; the path shards with no exchange)
# ---------------------------------------------------------------------------

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [ln.strip().split(", ") for ln in self.f.read().splitlines() if ln.strip()]
        self.f.close()
        os.unlink(self.f.name)
        return rows

    @staticmethod
    def summarise(rows, t0: float, t1: float):
        def ts(r):
            try:
                return time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                    float("0." + r[0].split(".")[1]) if "." in r[0] else 0.0
            except (ValueError, IndexError):
                return 0.0
        inside = [r for r in rows if len(r) >= 10 and t0 - 0.15 <= ts(r) <= t1 + 0.15]
        note = "samples inside the timed region"
        if not inside:
            inside = [r for r in rows if len(r) >= 10]
            note = "timed region shorter than the sampling period: samples from warm-up and timed steps"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        sm = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in inside for k in range(4) if r[6 + k].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# the CPU oracle as a baseline (bounded sample)
# ---------------------------------------------------------------------------

def oracle_inputs(w):
    """Seeded operands of the workload's shape for timing the oracle; the scale
    is that of a projection of N(0,1) states by N(0,0.02) weights."""
    s = 0.02 * math.sqrt(w.d_model)
    d = txl_inputs.draw_heads(w.B, w.H, w.L, w.M, w.dh, w.seed, std=s, bias_std=0.02)
    f = lambda t: t.double().numpy()
    return f(d["q"]), f(d["k"]), f(d["v"]), f(d["r"]), f(d["u"]), f(d["v_bias"])


def time_oracle(w, pairs_per_rep: int, min_seconds: float, max_reps: int):
    import oracle
    q, k, v, rel, u, vb = oracle_inputs(w)
    bh = list(range(min(pairs_per_rep, w.B * w.H)))
    reps, t = 0, 0.0
    while reps < max_reps and (reps == 0 or t < min_seconds):
        t0 = time.perf_counter()
        oracle.relattn(q, k, v, rel, u, vb, w.M, w.L, 1.0 / math.sqrt(w.dh), bh=bh)
        t += time.perf_counter() - t0
        reps += 1
    flops = 6.0 * w.L * w.K * w.dh * len(bh) * reps
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": round(t, 3),
            "sample": f"{w.name}: {len(bh)} of {w.B * w.H} (batch, head) slices per call, "
                      f"{reps} call(s), fp64 C oracle with OpenMP"}


def run_reference(args, world, rank):
    w = txl_inputs.WORKLOADS[txl_inputs.HEADLINE]
    if rank != 0:
        return
    import oracle
    cores = oracle.max_threads()
    pairs = max(1, min(w.B * w.H, cores))
    q, k, v, rel, u, vb = oracle_inputs(w)
    bh = list(range(pairs))
    run = lambda: oracle.relattn(q, k, v, rel, u, vb, w.M, w.L, 1.0 / math.sqrt(w.dh), bh=bh)
    t0 = time.perf_counter()
    run()
    t_step = time.perf_counter() - t0
    steps = max(1, min(args.steps, int(120.0 / max(t_step, 1e-3))))
    for _ in range(max(0, min(args.warmup, 3) - 1)):
        run()
    t0 = time.perf_counter()
    for _ in range(steps):
        run()
    t = time.perf_counter() - t0
    flops = 6.0 * w.L * w.K * w.dh * pairs * steps
    val = flops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "M": w.M, "K": w.K,
                   "dh": w.dh, "d_model": w.d_model,
                   "sample": f"{pairs} of {w.B * w.H} (batch, head) slices per step"},
        "tokens_per_s": pairs * w.L * steps / t / (w.H),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{pairs} (batch, head) slices of {w.name} per step, "
                                   f"{steps} steps (capped at ~120 s)"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling over disjoint units)."""
    return base + 1000 * rank


def build_operands(w, dev, rank=0):
    import torch
    import transformer_xl_relative_pos_gb300 as txl
    from transformer_xl_relative_pos_gb300 import model
    raw = txl_inputs.draw_layer(w, seed=rank_seed(w.seed, rank))
    h_ext = raw["h_ext"].to(dev)
    R = txl.rel_pos_emb(w.K, w.d_model, dtype=torch.float32, device=dev)
    q, k, v, r = model.attention_operands(h_ext, w.M, raw["W_q"].to(dev), raw["W_kE"].to(dev),
                                          raw["W_v"].to(dev), raw["W_kR"].to(dev), R, w.H,
                                          torch.bfloat16)
    h_seg = h_ext[:, w.M:].to(torch.bfloat16).contiguous()   # the segment's states [B, L, d]
    mem = h_ext[:, :w.M].to(torch.bfloat16).contiguous()     # a full memory [B, M, d]
    u = raw["u"].to(dev, torch.bfloat16)
    vb = raw["v_bias"].to(dev, torch.bfloat16)
    torch.cuda.synchronize()
    return {"q": q, "k": k, "v": v, "r": r, "u": u, "v_bias": vb, "h": h_seg, "mem": mem}


def run_e2e(w, dev, hs, r, u, vb, scale, ws, flops_step, n_steps):
    """End to end through the API, as a recurrent evaluation runs it (§3.2).

    The memory's projected keys and values stay on the device between segments,
    each in a window of a larger buffer (txl_kv_window_append / _advance), so
    the attention reads [memory ; segment] in place (txl_relattn_fwd_strided):
    nothing is concatenated.  Each step copies in, from pinned host buffers,
    only what is new (the segment's q, k, v and hidden states, one copy of one
    buffer), appends the segment to the k and v windows, attends over all
    K = M + L keys, advances the windows and the hidden-state memory ring
    (txl_mem_update), and reads the output back.  Two different host segments
    alternate.  The copies of step n+1 run on a copy stream while step n's
    kernels run (two device input sets), and each result is read back on a
    third stream.  Once the memories are full the device work of a step is
    replayed from a CUDA graph: the windows (capacity M + 25 L) and the ring
    both repeat their positions every 25 steps, so one graph per step of that
    cycle and input set is captured in step order.  After the timed steps the
    last output is checked against an attention over [memory ; segment] built
    on the host from the known segment sequence."""
    import torch
    import transformer_xl_relative_pos_gb300 as txl
    B, H, BH, L_, M_, dh_ = w.B, w.H, w.B * w.H, w.L, w.M, w.dh
    cyc = M_ // math.gcd(M_, L_)          # ring positions of the hidden-state memory
    C = M_ + cyc * L_                     # window capacity: the same cycle (>= 2M + L)
    assert C >= 2 * M_ + L_
    g = torch.Generator().manual_seed(123)
    # the segment's q, k, v [B, H, L, 64] and hidden states [B, L, d]: set 0 as
    # drawn for the step, set 1 a second, different segment
    segs = [{"q": hs["q"].cpu(), "k": hs["k"][:, :, M_:].cpu(), "v": hs["v"][:, :, M_:].cpu(),
             "h": hs["h"].cpu()}]
    segs.append({k2: (t.float() + 0.25 * torch.randn(t.shape, generator=g)).to(t.dtype)
                 for k2, t in segs[0].items()})
    layout, off = {}, 0
    for k2, t in segs[0].items():
        nb = t.numel() * t.element_size()
        layout[k2] = (off, nb, t.dtype, tuple(t.shape))
        off += (nb + 255) // 256 * 256
    h2d = off

    def views(flat):
        return {k2: flat[o:o + nb].view(dt).view(sh) for k2, (o, nb, dt, sh) in layout.items()}

    host_flat = [torch.empty(h2d, dtype=torch.uint8).pin_memory() for _ in range(2)]
    for j in range(2):
        for k2, t in views(host_flat[j]).items():
            t.copy_(segs[j][k2].contiguous())
    outs_h = [torch.empty(hs["out"].shape, dtype=hs["out"].dtype).pin_memory() for _ in range(2)]
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    dev_flat = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_in = [views(f) for f in dev_flat]
    dev_out = [torch.empty_like(hs["out"]) for _ in range(2)]
    kbuf = torch.empty(BH, C, dh_, dtype=torch.bfloat16, device=dev)
    vbuf = torch.empty_like(kbuf)
    h_ring = torch.empty_like(hs["mem"])
    k_win, v_win = txl.KVWindow(0, 0, C, M_), txl.KVWindow(0, 0, C, M_)
    h_st = txl.MemState(0, 0, M_)
    copy_s, comp_s, back_s = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_free = [torch.cuda.Event() for _ in range(2)]    # step's kernels done with its inputs
    in_ready = [torch.cuda.Event() for _ in range(2)]   # step's inputs copied
    out_ready = [torch.cuda.Event() for _ in range(2)]  # step's output written
    out_read = [torch.cuda.Event() for _ in range(2)]   # step's output read back
    for e in in_free + out_read:
        e.record(comp_s)

    def device_work(b):
        x = dev_in[b]
        m_cur = k_win.fill
        k_new = x["k"].view(BH, L_, dh_)
        v_new = x["v"].view(BH, L_, dh_)
        txl.kv_window_append(kbuf, k_win, k_new)
        txl.kv_window_append(vbuf, v_win, v_new)
        txl.relattn_fwd(x["q"], txl.kv_window_view(kbuf, k_win, L_, B, H),
                        txl.kv_window_view(vbuf, v_win, L_, B, H), r, u, vb, m_cur, scale,
                        out=dev_out[b], workspace=ws)
        txl.kv_window_advance(k_win, L_)
        txl.kv_window_advance(v_win, L_)
        txl.mem_update(h_ring, h_st, x["h"])

    graphs = {}  # step index within the cycle -> captured device work

    def e2e_step(i, cycle=None):
        b = i % 2
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(in_free[b])
            dev_flat[b].copy_(host_flat[b], non_blocking=True)
            in_ready[b].record(copy_s)
        with torch.cuda.stream(comp_s):
            comp_s.wait_event(in_ready[b])
            comp_s.wait_event(out_read[b])
            if cycle is None:
                device_work(b)
            else:
                graphs[i % cycle].replay()
            in_free[b].record(comp_s)
            out_ready[b].record(comp_s)
        with torch.cuda.stream(back_s):
            back_s.wait_event(out_ready[b])
            outs_h[b].copy_(dev_out[b], non_blocking=True)
            out_read[b].record(back_s)

    def drain():
        for s_ in (copy_s, comp_s, back_s):
            s_.synchronize()

    # Fill the memories from the host, and run eagerly until the windows have
    # moved back to their buffers' front once: from then on their positions
    # repeat every 25 steps (before, while M / L is not a whole number, they
    # follow a different sequence).  Then capture one graph per step of the
    # cycle, in step order (the host-side window and ring states advance as the
    # eager calls advance them).
    i, moved_back = 0, False
    while i < -(-M_ // L_) + 3 or not moved_back:
        full = k_win.fill == M_
        e2e_step(i)
        moved_back = moved_back or (full and k_win.start == L_)  # appended at the front
        i += 1
        assert i < 10 * cyc, "the windows never moved back"
    e2e_step(i)
    n_fill = i + 1
    drain()
    assert k_win.fill == M_ and v_win.fill == M_ and h_st.fill == M_
    cycle = 2 * cyc  # positions x the two input sets
    cap_s = torch.cuda.Stream()
    cap_s.wait_stream(comp_s)
    for i in range(n_fill, n_fill + cycle):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_s):
            with torch.cuda.graph(g_, stream=cap_s):
                device_work(i % 2)
        graphs[i % cycle] = g_
    comp_s.wait_stream(cap_s)
    for i in range(n_fill, n_fill + 3):
        e2e_step(i, cycle)
    drain()
    base_i = n_fill + 3
    t0 = time.perf_counter()
    for i in range(n_steps):
        e2e_step(base_i + i, cycle)
    drain()
    t_e2e = time.perf_counter() - t0
    # Check the last step independently: its memory is the newest M rows of the
    # k, v stream of all earlier segments (set (i % 2) at step i), its segment
    # the last one; attention over [memory ; segment] concatenated here.
    last = base_i + n_steps - 1
    need = -(-M_ // L_)
    kv = {}
    for name in ("k", "v"):
        hist = torch.cat([segs[i % 2][name] for i in range(last - need, last)], dim=2)
        kv[name] = torch.cat([hist[:, :, -M_:], segs[last % 2][name]], dim=2).to(dev)
    want = txl.relattn_fwd(segs[last % 2]["q"].to(dev), kv["k"], kv["v"], r, u, vb, M_, scale,
                           workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(dev_out[last % 2], want), "replayed step differs from the direct attention"
    assert torch.equal(outs_h[last % 2], want.cpu()), "host copy of the output differs"
    assert txl.device_status() == 0
    return {"value": flops_step * n_steps / t_e2e / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n_steps, "ms_per_step": 1e3 * t_e2e / n_steps,
            "inputs": "per step from pinned host memory: the segment's q, k, v [B, H, L, 64] and "
                      "hidden states [B, L, d_model], two different segments alternating; the "
                      "memory's k, v (M rows) stay on the device in windows filled from the host "
                      "by earlier steps",
            "device_work": "kv_window_append (k, v) + relattn_fwd over K = M + L keys read in "
                           "place (strided) + kv_window_advance + mem_update (h), replayed from "
                           "one CUDA graph per step of the 25-step cycle; the last output checked "
                           "equal to an attention over [memory ; segment] rebuilt on the host",
            "timing": "host clock around all steps (copies on their own streams), synchronized "
                      "on both sides"}


def run_ours(args, world, rank, local):
    import torch
    import transformer_xl_relative_pos_gb300 as txl

    w = txl_inputs.WORKLOADS[txl_inputs.HEADLINE]
    dev = torch.device("cuda", local)
    pk = peaks()
    base = build_operands(w, dev, rank)
    scale = 1.0 / math.sqrt(w.dh)
    ws = torch.empty(max(txl.workspace_size(w.B, w.H, w.L, w.dh, 8), 256), dtype=torch.uint8,
                     device=dev)
    sets = []
    for s in range(N_SETS):
        sets.append({
            "q": base["q"].clone(), "k": base["k"].clone(), "v": base["v"].clone(),
            "h": base["h"].clone(), "mem": base["mem"].clone(),
            "out": torch.empty_like(base["q"]),
            "out2": torch.empty_like(base["q"]),  # for steps of the second chain
            "st": txl.MemState(0, w.M, w.M),
        })
    r, u, vb = base["r"], base["u"], base["v_bias"]
    del base
    torch.cuda.synchronize()

    # Consecutive steps are independent batches (rotating input sets), so the
    # step graph runs them as two chains of attentions on two streams, steps
    # alternating: one step's first wave of blocks takes the SMs the other's
    # last wave leaves idle (256 blocks on 152 SMs).  The memory update of a step
    # is independent of its attention (it reads the segment's h and writes the
    # ring; the attention reads q, k, v and r) and runs on a third stream.  Each
    # step is forked from the launching stream; the graph joins every chain at
    # its end.  A dependent chain of calls (one layer's attention feeding the
    # next) gets none of this overlap: the line also reports the same steps on
    # one stream ("one_stream").
    chains = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    ws2 = torch.empty_like(ws)  # the second chain's split-key scratch
    side = torch.cuda.Stream(dev)
    forks = [torch.cuda.Event() for _ in range(N_SETS)]

    def step(i, streams=2):
        s = sets[i % N_SETS]
        fork = forks[i % N_SETS]
        main = torch.cuda.current_stream(dev)
        fork.record(main)
        att = chains[i % 2] if streams == 2 else main
        att.wait_event(fork)
        side.wait_event(fork)
        # each chain writes its own outputs (steps i and i + 3 share an input
        # set and may run at the same time on the two chains)
        second = streams == 2 and i % 2 == 1
        out = s["out2"] if second else s["out"]
        with torch.cuda.stream(att):
            txl.relattn_fwd(s["q"], s["k"], s["v"], r, u, vb, w.M, scale, out=out,
                            workspace=ws2 if second else ws)
        with torch.cuda.stream(side):
            txl.mem_update(s["mem"], s["st"], s["h"])

    # Kernel launches per step: the attention (plus a merge when its key range
    # is split) and the memory update.
    kern, n_split = txl.relattn_plan(w.B, w.H, w.M, w.L, workspace_bytes=ws.numel())
    launches_per_step = 2 + (1 if n_split > 1 else 0)

    for i in range(max(args.warmup, 3)):
        step(i)
    for s_ in chains + [side]:
        torch.cuda.current_stream(dev).wait_stream(s_)
    torch.cuda.synchronize()
    assert txl.device_status() == 0

    K = max(1, args.steps)
    if K <= 2 * GRAPH_CHUNK:
        chunk, reps = K, 1
    else:
        chunk = GRAPH_CHUNK
        reps = max(1, round(K / GRAPH_CHUNK))
        K = chunk * reps
    def capture(streams):
        g = torch.cuda.CUDAGraph()
        cap_stream = torch.cuda.Stream(dev)
        cap_stream.wait_stream(torch.cuda.current_stream(dev))
        for s_ in chains + [side]:
            s_.wait_stream(cap_stream)
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(g, stream=cap_stream):
                for i in range(chunk):
                    step(i, streams)
                for s_ in (chains if streams == 2 else []) + [side]:
                    cap_stream.wait_stream(s_)  # join every chain
        torch.cuda.current_stream(dev).wait_stream(cap_stream)
        return g

    g = capture(2)
    g.replay()  # untimed replay: graph upload and warm caches
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    clocks = ClockSampler.summarise(sampler.stop(), wall0, wall1) if sampler else None
    t_ms = max_over_ranks(e0.elapsed_time(e1), world)
    status = txl.device_status()

    # The attention kernel's launch time, right after the timed region: a graph
    # of back-to-back attention launches on the same rotating input sets, in
    # the launch configuration of the step, timed as a whole with CUDA events
    # on the launching stream.  (An event recorded inside a graph costs several
    # microseconds, so events around each launch would time the events too.)
    n_attn = max(3 * N_SETS, min(chunk, 300) // N_SETS * N_SETS)
    attn_timing = (f"graph of {n_attn} back-to-back attention launches on the {N_SETS} rotating "
                   f"input sets, replayed right after the timed region, CUDA events around the replay")
    ga = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        with torch.cuda.graph(ga, stream=cs):
            for i in range(n_attn):
                s_ = sets[i % N_SETS]
                txl.relattn_fwd(s_["q"], s_["k"], s_["v"], r, u, vb, w.M, scale,
                                out=s_["out"], workspace=ws)
    torch.cuda.current_stream(dev).wait_stream(cs)
    ga.replay()
    torch.cuda.synchronize()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_.record(stream)
    ga.replay()
    b_.record(stream)
    torch.cuda.synchronize()
    attn_ms = a_.elapsed_time(b_) / n_attn
    del ga

    # The same K steps on one stream (each step's attention after the previous
    # one's), timed the same way: what a chain of dependent calls gets.
    g1 = capture(1)
    g1.replay()
    torch.cuda.synchronize()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_.record(stream)
    for _ in range(reps):
        g1.replay()
    b_.record(stream)
    torch.cuda.synchronize()
    one_ms = max_over_ranks(a_.elapsed_time(b_), world)
    del g1

    # The sinusoid table kernel, per layer (outside the step): graph-replayed.
    R_buf = torch.empty(w.K, w.d_model, dtype=torch.float32, device=dev)
    gr = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cs):
        with torch.cuda.graph(gr, stream=cs):
            for _ in range(50):
                txl.rel_pos_emb(w.K, w.d_model, out=R_buf)
    torch.cuda.current_stream(dev).wait_stream(cs)
    gr.replay()
    torch.cuda.synchronize()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_.record(stream)
    gr.replay()
    b_.record(stream)
    torch.cuda.synchronize()
    relpos_us = a_.elapsed_time(b_) * 1e3 / 50
    del R_buf

    flops_step = w.flops()
    value = flops_step * K * world / (t_ms * 1e-3) / 1e12
    one_stream = {"ms_per_step": one_ms / K,
                  "value": flops_step * K * world / (one_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                  "note": "the same steps with every attention on one stream, one after another"}
    tokens = w.B * w.L * K * world / (t_ms * 1e-3)
    # "useful" work: only the scores a query may see (j <= M + i), i.e.
    # L*M + L(L+1)/2 of the L*K pairs per head
    visible = (w.L * w.M + w.L * (w.L + 1) // 2) / (w.L * (w.M + w.L))

    # ---- end to end through the public API with host buffers ----------------
    e2e = None
    if rank == 0 and args.e2e_steps > 0:
        e2e = run_e2e(w, dev, sets[0], r, u, vb, scale, ws, flops_step, args.e2e_steps)

    if rank != 0:
        return
    # ---- roofline of the attention kernel -----------------------------------
    bytes_alg = 2 * (w.B * w.H * w.L * w.dh * 2 + 2 * w.B * w.H * w.K * w.dh) + w.H * w.K * w.dh * 2
    attn_s = attn_ms * 1e-3
    achieved_gbs = bytes_alg / attn_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved_gbs / pk["hbm_gbs"], "traffic": profiled_traffic(w.name),
                "kernel": "relattn_fwd_tc_kernel", "launch_us": attn_ms * 1e3,
                "timing": attn_timing,
                "tensor_tflops": flops_step / attn_s / 1e12,
                "tensor_frac": flops_step / attn_s / 1e12 / pk["bf16_tflops"],
                "peak_source": pk["source"] + " (MEASURED_PEAKS.json burst figures)"}
    cpu = None
    if not args.no_cpu_baseline:
        cpu = time_oracle(w, pairs_per_rep=w.B * w.H, min_seconds=10.0, max_reps=6)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": t_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "M": w.M, "K": w.K,
                   "dh": w.dh, "d_model": w.d_model,
                   "step": "relattn_fwd + mem_update over one batch (table R and r built once "
                           "per layer, outside the step)",
                   "streams": "steps are independent batches: their attentions alternate between "
                              "two streams (one step's first wave fills the SMs the other's last "
                              "wave leaves idle), memory updates on a third",
                   "l2": f"{N_SETS} rotating input sets (>2x L2 of traffic between reuses)",
                   "launch": f"CUDA graph of {chunk} steps x {reps} replays"},
        "tokens_per_s": tokens,
        "pct_bf16_peak": 100.0 * value / pk["bf16_tflops"],
        "useful_tflops": value * visible,
        "attn_us": attn_ms * 1e3,
        "one_stream": one_stream,
        "rel_pos_emb_us": relpos_us,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "device_status": status,
        "roofline": roofline,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# Evaluation speed ("Transformer-XL: Attentive Language Models Beyond a
# Fixed-Length Context", §4.5, Table 9; the vanilla evaluation procedure is
# §3.1): for each new token the vanilla model processes a whole window of A
# positions from scratch (L = A queries, no memory), while Transformer-XL
# reuses the cached states (L = 1 new query against M = A - 1 memory rows, or
# a segment of 128 queries against A - 128 rows, per token / 128).  Attention of
# one layer only, random bf16 operands, H = 16 heads of 64; times graph-replayed.
TABLE9_PAPER = {800: 363, 1800: 773, 2800: 1409, 3800: 1874}


def attn_call_us(B, H, L, M, reps=10, per=20, n_sets=1):
    """Device time of one txl_relattn_fwd call (graph-replayed), random bf16
    operands; with n_sets > 1 the calls rotate over that many input sets (k, v
    and the table larger than L2 in total keeps the reads in HBM)."""
    import torch
    import transformer_xl_relative_pos_gb300 as txl
    dev = torch.device("cuda", 0)
    K = M + L
    g = torch.Generator(device=dev).manual_seed(B * 7919 + L * 31 + M)
    mk = lambda *sh: (torch.randn(*sh, device=dev, generator=g) * 0.5).to(torch.bfloat16)
    sets = [(mk(B, H, L, 64), mk(B, H, K, 64), mk(B, H, K, 64), mk(H, K, 64)) for _ in range(n_sets)]
    u, vb = mk(H, 64) * 0.2, mk(H, 64) * 0.2
    out = torch.empty(B, H, L, 64, device=dev, dtype=torch.bfloat16)
    ws = torch.empty(max(txl.workspace_size(B, H, L, 64, 64), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()

    def call(i):
        q, k, v, r = sets[i % n_sets]
        txl.relattn_fwd(q, k, v, r, u, vb, M, 0.125, out=out, workspace=ws)

    with torch.cuda.stream(stream):
        for i in range(3):
            call(i)
    torch.cuda.synchronize()
    per = max(per, n_sets) // n_sets * n_sets
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(per):
            call(i)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    assert txl.device_status() == 0
    return e0.elapsed_time(e1) * 1e3 / (reps * per)


def run_table9(args):
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for B in (1, 16):
        for A in sorted(TABLE9_PAPER):
            vanilla = attn_call_us(B, 16, A, 0)
            xl_tok = attn_call_us(B, 16, 1, A - 1)
            xl_seg = attn_call_us(B, 16, 128, A - 128) / 128
            print(json.dumps({"table9": {
                "attn_len": A, "B": B, "H": 16, "d_head": 64, "dtype": "bf16",
                "vanilla_us_per_token": vanilla, "xl_decode_us_per_token": xl_tok,
                "xl_segment128_us_per_token": xl_seg,
                "slowdown_vs_decode": vanilla / xl_tok, "slowdown_vs_segment128": vanilla / xl_seg,
                "paper_slowdown": TABLE9_PAPER[A],
                "note": "one attention layer; the paper's ratio is for the whole model"}}), flush=True)


# Decode steps (one to eight new tokens against a long memory), H = 16 heads of
# 64: the memory lengths of the long-memory evaluation (M = 1600 and 3800).
DECODE_SHAPES = [(8, L, 3800) for L in range(1, 9)] + [
    (16, 1, 1600), (16, 6, 1600), (16, 8, 1600), (64, 1, 3800), (64, 6, 3800), (64, 8, 3800),
    (1, 1, 3800), (1, 6, 3800), (1, 8, 12000), (2, 6, 800)]


def run_decode(args):
    """Graph-replayed time and achieved HBM bandwidth of decode-shaped calls
    (L new queries per sequence against M cached positions)."""
    import torch
    import transformer_xl_relative_pos_gb300 as txl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk = peaks()
    shapes = [tuple(int(x) for x in s.split(",")) for s in args.shapes] if args.shapes else DECODE_SHAPES
    H = 16
    for B, L, M in shapes:
        K = M + L
        nbytes = 2 * (2 * B * H * K * 64 + H * K * 64 + 2 * B * H * L * 64)  # k, v, r, q, out (bf16)
        n_sets = max(1, min(3, -(-3 * 126 * 2 ** 20 // nbytes)))  # > L2 of traffic between reuses
        us = attn_call_us(B, H, L, M, reps=args.calls, per=30, n_sets=n_sets)
        gbs = nbytes / (us * 1e-6) / 1e9
        kernel, splits = txl.relattn_plan(B, H, M, L, workspace_bytes=txl.workspace_size(B, H, L, 64, 64))
        print(json.dumps({"decode": {
            "B": B, "H": H, "L": L, "M": M, "dtype": "bf16", "us_per_call": us,
            "algorithmic_bytes": nbytes, "achieved_gbs": gbs, "peak_gbs": pk["hbm_gbs"],
            "hbm_frac": gbs / pk["hbm_gbs"], "input_sets": n_sets,
            "path": {"decode": "decode kernel (CUDA cores)", "decode_mma": "decode kernel (warp MMAs)",
                     "tc": "tensor-core kernel"}[kernel],
            "splits": splits}}), flush=True)


def run_configs(args):
    """Graph-replayed attention calls of every bf16 workload shape (random
    operands, rotating input sets larger than L2): TFLOP/s, fraction of the
    bf16 peak and HBM bandwidth per shape."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk = peaks()
    for name, w in txl_inputs.WORKLOADS.items():
        if w.dtype != "bf16" or name.startswith("c5"):
            continue  # c5 is the stack; its attention call is c2's shape
        if args.workload and name not in args.workload:
            continue
        K = w.M + w.L
        nbytes = 2 * (2 * w.B * w.H * w.L * 64 + 2 * w.B * w.H * K * 64 + w.H * K * 64)
        n_sets = max(1, min(3, -(-3 * 126 * 2 ** 20 // nbytes)))
        us = attn_call_us(w.B, w.H, w.L, w.M, reps=args.calls, per=30, n_sets=n_sets)
        us_hot = attn_call_us(w.B, w.H, w.L, w.M, reps=args.calls, per=30, n_sets=1)
        tflops = w.flops() / (us * 1e-6) / 1e12
        print(json.dumps({"config": {
            "workload": name, "B": w.B, "H": w.H, "L": w.L, "M": w.M, "dtype": "bf16",
            "us_per_call": us, "tflops": tflops, "pct_bf16_peak": 100.0 * tflops / pk["bf16_tflops"],
            "achieved_gbs": nbytes / (us * 1e-6) / 1e9, "hbm_frac": nbytes / (us * 1e-6) / 1e9 / pk["hbm_gbs"],
            "input_sets": n_sets, "l2": "cold: calls rotate over the input sets",
            "us_per_call_l2_hot": us_hot,
            "tflops_l2_hot": w.flops() / (us_hot * 1e-6) / 1e12}}), flush=True)


def run_project(args):
    """Graph-replayed time of one layer's projections of a segment at the
    12-layer stream's shape (B=16, L=M=512, d=512, H=8): txl_qkv_project (q, k,
    v into q and the window, the memory update) against the calls it replaces
    (torch GEMM + head-major permutation + txl_kv_window_append +
    txl_mem_update) and against the GEMM alone."""
    import torch
    import transformer_xl_relative_pos_gb300 as txl
    from transformer_xl_relative_pos_gb300.model import project_stacked
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w_ = txl_inputs.WORKLOADS["c5_stack12_L512_M512"]
    B, H, L, M, d = w_.B, w_.H, w_.L, w_.M, w_.d_model
    C = M + 2 * L
    g = torch.Generator(device=dev).manual_seed(0)
    h = torch.randn(B, L, d, device=dev, generator=g).to(torch.bfloat16)
    W = (torch.randn(3 * H * 64, d, device=dev, generator=g) * d ** -0.5).to(torch.bfloat16)
    kv = torch.zeros(2 * B * H, C, 64, dtype=torch.bfloat16, device=dev)
    mem = torch.zeros(B, M, d, dtype=torch.bfloat16, device=dev)
    q = torch.empty(B, H, L, 64, dtype=torch.bfloat16, device=dev)

    def fused():
        txl.qkv_project(h, W, kv, txl.KVWindow(0, M, C, M), q=q, mem=mem,
                        mem_state=txl.MemState(0, M, M))

    def unfused():
        win = txl.KVWindow(0, M, C, M)
        qkv = project_stacked(h, W, 3, H)
        txl.kv_window_append(kv, win, qkv[1:].view(2 * B * H, L, 64))
        txl.mem_update(mem, txl.MemState(0, M, M), h)

    def gemm_only():
        torch.matmul(h, W.t())

    flops = 2.0 * B * L * 3 * H * 64 * d
    for name, fn in (("qkv_project", fused), ("unfused", unfused), ("library_gemm_only", gemm_only)):
        s_ = torch.cuda.Stream(dev)
        with torch.cuda.stream(s_):
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s_):
            for _ in range(20):
                fn()
        gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_)
        with torch.cuda.stream(s_):
            for _ in range(max(1, args.calls)):
                gr.replay()
        e1.record(s_)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (20 * max(1, args.calls))
        print(json.dumps({"project": {"op": name, "B": B, "L": L, "d_model": d, "H": H,
                                      "us_per_call": us, "tflops": flops / (us * 1e-6) / 1e12}}),
              flush=True)
    assert txl.device_status() == 0


def run_stack(args):
    """Per-segment time of the streaming stack on the 12-layer, 16-segment
    workload (B=16, H=8, L=M=512, d=512), memories full, with and without the
    cached projected memory keys/values, launched eagerly or replayed from CUDA
    graphs.  Torch does the projections, LayerNorm and feed-forward; the
    kernels do the table, the attention and the rings."""
    import torch
    from transformer_xl_relative_pos_gb300.model import XLStack
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = txl_inputs.WORKLOADS["c5_stack12_L512_M512"]
    params = txl_inputs.draw_stack(w)
    tokens = params["tokens"].to(dev)
    n_seg = tokens.shape[0]
    for graphs, cache_kv in ((False, True), (False, False), (True, True), (True, False)):
        stack = XLStack(params, w.H, w.M, dev, torch.bfloat16, cache_kv=cache_kv, graphs=graphs)
        # Memories are full after the first segment (L = M); with graphs one is
        # captured per distinct ring and window position, from the third segment
        # on (one position for the rings, two for the windows of capacity
        # M + 2L): the warm-up covers them all, so no capture falls in the
        # timed segments.  Segments cycle through the workload's 16.
        n_warm = 3 + 4
        for s_ in range(n_warm):
            stack.segment(tokens[s_ % n_seg])
        torch.cuda.synchronize()
        n_graphs = len(stack._graphs)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        n_timed = n_seg
        for s_ in range(n_warm, n_warm + n_timed):
            stack.segment(tokens[s_ % n_seg])
        e1.record()
        torch.cuda.synchronize()
        assert len(stack._graphs) == n_graphs, "a graph was captured inside the timed segments"
        ms = e0.elapsed_time(e1) / n_timed
        print(json.dumps({"stack": {
            "workload": w.name, "layers": len(params["layers"]), "B": w.B, "H": w.H, "L": w.L,
            "M": w.M, "d_model": w.d_model, "cache_kv": cache_kv, "cuda_graphs": graphs,
            "graphs": n_graphs, "segments_timed": n_timed,
            "ms_per_segment": ms, "tokens_per_s": w.B * w.L / (ms * 1e-3)}}), flush=True)


def bwd_tile_visits(B, H, L, M, T=64):
    """64 x 64 pair tiles each launch of txl_relattn_bwd visits (the kernels'
    loop bounds: key tiles up to the last key a chunk sees, query chunks from
    the first that sees a key tile or reaches a distance tile)."""
    K = M + L
    n_chunks = -(-L // T)
    rows_keys = sum(-(-min(K, M + i0 + T) // T) for i0 in range(0, L, T))
    keys_rows = sum(len(range(max(0, j0 - M) // T * T, L, T)) for j0 in range(0, K, T))
    dist_rows = B * sum(len(range(max(0, d0 - M) // T * T, L, T)) for d0 in range(0, K, T))
    v = {"stats": B * H * rows_keys, "dr": H * dist_rows, "chunks": B * H * n_chunks}
    if n_chunks <= 2:  # one pass for dq, dk and dv
        v["dqkv"] = B * H * rows_keys
    else:
        v["dq"], v["dkv"] = B * H * rows_keys, B * H * keys_rows
    return v


def run_bwd(args):
    """Graph-replayed time of one backward call (txl_relattn_bwd) at the headline
    shape (or the --workload named), over rotating input sets (k, v, q and dout;
    at least 160 MB together, more than L2 holds).  Reports the tensor-core FLOPs
    the kernels execute (warp-level bf16 MMAs, fp32
    accumulation: scores recomputed per pass, the position terms as 64 x 128
    window products, the products with g and P twice for their bf16 head and
    rest) against the measured bf16 peak, and the rate of the backward's own
    FLOPs (twice the forward's: dP, dv, and the gradients of the content and
    position scores)."""
    import torch
    import transformer_xl_relative_pos_gb300 as txl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = txl_inputs.WORKLOADS[args.workload[0] if args.workload else txl_inputs.HEADLINE]
    if w.dtype != "bf16":
        raise SystemExit(f"--bwd: {w.name} is {w.dtype}; the backward takes bf16 inputs")
    B, H, L, M = w.B, w.H, w.L, w.M
    K = M + L
    g = torch.Generator(device=dev).manual_seed(0)
    mk = lambda *sh: (torch.randn(*sh, device=dev, generator=g) * 0.6).to(torch.bfloat16)
    set_bytes = 2 * 64 * B * H * (2 * L + 2 * K)
    n_sets = max(2, math.ceil(160e6 / set_bytes))
    sets = [(mk(B, H, L, 64), mk(B, H, K, 64), mk(B, H, K, 64), mk(B, H, L, 64)) for _ in range(n_sets)]
    r, u, vb = mk(H, K, 64), mk(H, 64) * 0.5, mk(H, 64) * 0.5
    f32 = lambda *sh: torch.empty(*sh, dtype=torch.float32, device=dev)
    grads = (f32(B, H, L, 64), f32(B, H, K, 64), f32(B, H, K, 64), f32(H, K, 64), f32(H, 64),
             f32(H, 64))
    ws = torch.empty(max(txl.bwd_workspace_size(B, H, L, M), 256), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(64)

    def call(i):
        q, k, v, dout = sets[i % n_sets]
        txl.relattn_bwd(q, k, v, r, u, vb, dout, M, scale, grads=grads, workspace=ws)

    st = torch.cuda.Stream(dev)
    with torch.cuda.stream(st):
        for i in range(3):
            call(i)
    torch.cuda.synchronize()
    per = 10
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=st):
        for i in range(per):
            call(i)
    gr.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    with torch.cuda.stream(st):
        for _ in range(max(1, args.calls)):
            gr.replay()
    e1.record(st)
    torch.cuda.synchronize()
    assert txl.device_status() == 0
    us = e0.elapsed_time(e1) * 1e3 / (per * max(1, args.calls))
    visits = bwd_tile_visits(B, H, L, M)
    T = 64
    # launches per call: segments of at most two row chunks take the two-chunk
    # statistics and one-pass dq/dk/dv kernels over key splits (the count that
    # fills the SMs' waves best, at most 8), each followed by an ordered merge
    # when split; longer ones the per-chunk statistics, dq and dk/dv kernels;
    # then the table gradient and the bias sums
    if -(-L // T) <= 2:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        n_splits, best = 1, 0.0
        for sp in range(1, min(8, -(-K // T)) + 1):
            eff = B * H * sp / (math.ceil(B * H * sp / sms) * sms)
            if eff > best + 0.03:
                best, n_splits = eff, sp
        launches = 4 + (2 if n_splits > 1 else 0)
    else:
        launches = 5
    # tile multiply-adds: stats q.k, dout.v (64^3 each), the q.r window (2 x 64^3);
    # dq adds g.k and the window-ordered g.r (head and rest: 2 x 3 x 64^3);
    # dk/dv add P^T dout and g^T q (2 x 2 x 64^3); the one-pass dq / dk / dv
    # launch of short segments: scores, dq's and dk/dv's products; the table
    # tile: g^T q from the stored g, read along its diagonals (2 x 64^3)
    mac_tile = {"stats": 4 * T ** 3, "dq": 10 * T ** 3, "dkv": 8 * T ** 3, "dr": 2 * T ** 3,
                "dqkv": 14 * T ** 3}
    executed = 2.0 * sum(visits[k] * mac_tile[k] for k in mac_tile if k in visits)
    pk = peaks()
    useful = 2.0 * 6.0 * L * K * 64 * B * H
    print(json.dumps({"bwd": {
        "workload": w.name, "B": B, "H": H, "L": L, "M": M, "us_per_call": round(us, 2),
        "input_sets": n_sets, "input_mb": round(n_sets * set_bytes / 1e6, 1),
        "executed_tensor_gflop": round(executed / 1e9, 1),
        "executed_tflops": round(executed / (us * 1e-6) / 1e12, 2),
        "bf16_peak_tflops": pk["bf16_tflops"], "peak_source": pk["source"],
        "tensor_frac": round(executed / (us * 1e-6) / 1e12 / pk["bf16_tflops"], 4),
        "useful_gflop": round(useful / 1e9, 1),
        "useful_tflops": round(useful / (us * 1e-6) / 1e12, 2),
        "tile_visits": visits, "launches": launches,
        # g of every pair, fp32: written by the dq pass, read by the table gradient
        "g_stored_mb": round(B * H * L * K * 4 / 1e6, 1)}}), flush=True)


def main():
    args = parse_args()
    if args.bwd:
        run_bwd(args)
        return
    if args.stack:
        run_stack(args)
        return
    if args.project:
        run_project(args)
        return
    if args.table9:
        run_table9(args)
        return
    if args.decode:
        run_decode(args)
        return
    if args.configs:
        run_configs(args)
        return
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
