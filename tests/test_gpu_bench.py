"""bench.py on the GPU: our arm prints one JSON line with the benchmark
contract's keys, the roofline of the attention kernel, and an end-to-end leg
whose graph-replayed steps were checked against an eager step inside the run
(bench.py asserts that before it prints)."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_bench_line_contract_and_end_to_end_leg():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "200",
                          "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "20"],
                         cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-3000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "clocks",
                "e2e", "gpu_launches", "roofline"):
        assert key in line, key
    assert line["value"] > 0 and line["n_gpus"] == 1 and line["device_status"] == 0
    assert line["config"]["workload"] == "c3_word_large_L128_M1600"
    # per step: the attention (plus a merge when its key range is split) and the
    # memory update; the table is built once per layer, outside the step
    assert line["gpu_launches"] >= 2 * line["steps"]
    assert line["rel_pos_emb_us"] > 0
    # the same steps with all attentions on one stream are reported beside the
    # two-chain figure (consecutive steps are independent batches)
    one = line["one_stream"]
    assert one["value"] > 0 and one["ms_per_step"] > 0
    roof = line["roofline"]
    assert roof["kernel"] == "relattn_fwd_tc_kernel" and 0 < roof["frac"] and roof["peak"] > 0
    e2e = line["e2e"]
    # one segment in per step: q, k, v [16, 16, 128, 64] and h [16, 128, 1024], bf16
    assert e2e["h2d_bytes_per_step"] == 4 * 16 * 128 * 1024 * 2
    assert e2e["d2h_bytes_per_step"] == 16 * 16 * 128 * 64 * 2
    assert e2e["value"] > 0 and e2e["steps"] == 20
