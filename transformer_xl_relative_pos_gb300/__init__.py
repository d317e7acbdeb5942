"""GB300 (sm_103a) Transformer-XL relative-position attention.

Thin Python binding over the C ABI of ``libtxl_gb300.so`` (``include/txl.h``).
Every function here only marshals arguments (tensor pointers, sizes, the
current CUDA stream) and raises on a non-zero status; all computation runs in
the library's CUDA kernels.  There is no CPU fallback: without the built
library every call raises.

Functions follow "Transformer-XL: Attentive Language Models Beyond a
Fixed-Length Context" (§3.2 segment-level recurrence, §3.3 relative score and
N-layer summary, Appendix B reversed table and shift):

  rel_pos_emb     sinusoid table R in Appendix B's reversed row order
  relattn_fwd     fused relative-position attention over [memory ; segment]
  relattn_plan    which kernel and key split relattn_fwd would use
  mem_concat      extended context [SG(m) o h] from the ring-buffer memory
  mem_update      advance the memory to the newest M states
  kv_window_*     a memory kept as a window of a larger buffer, read in place
                  by relattn_fwd (k, v as strided views)
  qkv_project     one layer's q, k, v projections written into q and the k / v
                  window, with the memory update, in one launch
  relattn_bwd     gradients of relattn_fwd for one segment (training within a
                  segment, the memory SG(m))
"""

from __future__ import annotations

from ._lib import (  # noqa: F401
    F32,
    BF16,
    KVWindow,
    MemState,
    TxlError,
    bwd_workspace_size,
    debug_checks,
    debug_index_probe,
    debug_wait_timeout,
    device_status,
    kv_window_advance,
    kv_window_append,
    kv_window_view,
    lib,
    lib_path,
    mem_concat,
    mem_update,
    qkv_project,
    rel_pos_emb,
    relattn_bwd,
    relattn_fwd,
    relattn_fwd_noalloc,
    relattn_plan,
    set_wait_limit_ns,
    status_string,
    version,
    workspace_size,
)
