"""txl_relattn_fwd_noalloc: attention for callers that cannot allocate.

Some callers cannot allocate device memory when they run attention: plugins of
inference engines whose execute step must not allocate, and runtimes whose
device-memory budget is fixed at start-up.  For them the library offers an
entry point whose split-key partial results live in a scratch array built into
the library instead of a caller workspace.  These tests check, through the C
ABI, that it gives the same output as the workspace entry point on two calls in
a row (the second call finds the first call's leftovers in the shared scratch),
for a tensor-core split and for a decode split merged through the scratch; that
one split case also matches the fp64 oracle directly; and that a split larger
than the scratch is refused.

This file is collected last on purpose: it depends on nothing the other tests
leave behind and passes alone in a fresh process as well.
"""

import math

import pytest
import torch

import transformer_xl_relative_pos_gb300 as txl
from parity import TOL_BF16, TOL_BF16_RMS, compare, dev, heads_case, run_oracle

pytestmark = pytest.mark.gpu


def _operands(case):
    d = dev()
    return {k: t.to(d).contiguous() for k, t in case.items()}


# (B, H, L, M, n_splits, kernel): a tensor-core split, the automatic choice, and
# decode calls (both kernels) with more key ranges than one thread-block cluster
# merges, so that their partials go through the scratch and the merge kernel.
CASES = [(2, 3, 130, 900, 3, "tc"), (2, 3, 130, 900, 0, "tc"), (2, 3, 3, 2000, 12, "decode_mma"),
         (2, 3, 1, 2000, 12, "decode")]


@pytest.mark.parametrize("B,H,L,M,n_splits,kernel", CASES)
def test_noalloc_matches_workspace_entry_point_twice(B, H, L, M, n_splits, kernel):
    case = heads_case(B, H, L, M, seed=41 + L)
    t = _operands(case)
    scale = 1.0 / math.sqrt(64)
    ws_bytes = txl.workspace_size(B, H, L, 64, max(n_splits, 8))
    assert txl.relattn_plan(B, H, M, L, n_splits=n_splits, workspace_bytes=ws_bytes)[0] == kernel
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev())
    ref, ref_lse = txl.relattn_fwd(t["q"], t["k"], t["v"], t["r"], t["u"], t["v_bias"], M, scale,
                                   lse=True, n_splits=n_splits, workspace=ws)
    for _ in range(2):
        out, lse = txl.relattn_fwd_noalloc(t["q"], t["k"], t["v"], t["r"], t["u"], t["v_bias"],
                                           M, scale, lse=True, n_splits=n_splits)
        torch.cuda.synchronize()
        assert txl.device_status() == 0
        compare(out.float().cpu().numpy(), ref.float().cpu().numpy(), TOL_BF16, what="out")
        compare(lse.cpu().numpy(), ref_lse.cpu().numpy(), TOL_BF16, what="lse")


def test_noalloc_split_matches_oracle():
    # The same entry point checked against the fp64 oracle on its own, with the
    # key range of every head split over three blocks.
    B, H, L, M = 2, 2, 130, 700
    case = heads_case(B, H, L, M, seed=59)
    t = _operands(case)
    out, lse = txl.relattn_fwd_noalloc(t["q"], t["k"], t["v"], t["r"], t["u"], t["v_bias"], M,
                                       0.125, lse=True, n_splits=3)
    torch.cuda.synchronize()
    assert txl.device_status() == 0
    want, want_lse = run_oracle(case, M, 0.125)
    compare(out.float().cpu().numpy(), want, TOL_BF16, TOL_BF16_RMS, what="noalloc split 3")
    compare(lse.cpu().numpy(), want_lse, TOL_BF16, what="noalloc lse split 3")


def test_noalloc_refuses_split_beyond_scratch():
    # 16 x 16 heads of 128 queries split 8 ways needs about 68 MB of partials.
    B, H, L, M = 16, 16, 128, 1600
    assert txl.workspace_size(B, H, L, 64, 8) > 32 * 1024 * 1024
    q = torch.empty(B, H, L, 64, dtype=torch.bfloat16, device=dev())
    kv = torch.empty(B, H, M + L, 64, dtype=torch.bfloat16, device=dev())
    r = torch.empty(H, M + L, 64, dtype=torch.bfloat16, device=dev())
    uv = torch.empty(H, 64, dtype=torch.bfloat16, device=dev())
    with pytest.raises(txl.TxlError) as e:
        txl.relattn_fwd_noalloc(q, kv, kv, r, uv, uv, M, 0.125, n_splits=8)
    assert e.value.status == -7
