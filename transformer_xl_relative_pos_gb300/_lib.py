"""ctypes binding of the C ABI in ``include/txl.h`` (argument marshalling only)."""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

F32 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None

_c_int, _c_size, _c_p, _c_float, _c_u64 = (ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p,
                                           ctypes.c_float, ctypes.c_uint64)


class TxlError(RuntimeError):
    """A non-zero txl_status returned by the library."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class KVWindow(ctypes.Structure):
    """txl_kv_window: host-side state of a memory kept as a contiguous window of
    a larger buffer [planes, capacity, d] (capacity >= 2 M + L)."""

    _fields_ = [("start", ctypes.c_int), ("fill", ctypes.c_int), ("capacity", ctypes.c_int),
                ("M", ctypes.c_int)]

    def __repr__(self):
        return (f"KVWindow(start={self.start}, fill={self.fill}, capacity={self.capacity}, "
                f"M={self.M})")


class MemState(ctypes.Structure):
    """txl_mem_state: host-side ring-buffer state of one layer's memory."""

    _fields_ = [("head", ctypes.c_int), ("fill", ctypes.c_int), ("capacity", ctypes.c_int)]

    def __repr__(self):
        return f"MemState(head={self.head}, fill={self.fill}, capacity={self.capacity})"


def _debug() -> bool:
    return os.environ.get("TXL_DEBUG_LIB") == "1"


def lib_path() -> str:
    return _build.DEBUG_LIB_PATH if _debug() else _build.LIB_PATH


def lib():
    """Load ``libtxl_gb300.so`` (with TXL_DEBUG_LIB=1 in the environment: the
    debug build ``libtxl_gb300_debug.so``); build it first when the sources are
    newer.

    Raises if it cannot be built or loaded: nothing falls back to another
    implementation."""
    global _lib
    with _lock:
        if _lib is None:
            if os.environ.get("TXL_NO_BUILD") == "1":
                path = lib_path()
            else:
                path = _build.build(debug=_debug())
            if not os.path.exists(path):
                raise TxlError(-5, f"CUDA library missing: {path}")
            L = ctypes.CDLL(path)
            sig = {
                "txl_status_string": (ctypes.c_char_p, [_c_int]),
                "txl_version": (_c_int, []),
                "txl_rel_pos_emb": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_p]),
                "txl_relattn_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
                "txl_relattn_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                              _c_int, _c_size, ctypes.POINTER(_c_int),
                                              ctypes.POINTER(_c_int)]),
                "txl_relattn_fwd": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p, _c_p,
                                             _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                             _c_int, _c_int, _c_p, _c_size, _c_p]),
                "txl_relattn_fwd_strided": (_c_int, [_c_p, _c_p, _c_p, ctypes.c_longlong, _c_p,
                                                     _c_int, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int,
                                                     _c_int, _c_int, _c_int, _c_float, _c_int,
                                                     _c_int, _c_p, _c_size, _c_p]),
                "txl_kv_window_append": (_c_int, [_c_p, ctypes.POINTER(KVWindow), _c_p, _c_int,
                                                  _c_int, _c_int, _c_int, _c_p]),
                "txl_kv_window_advance": (_c_int, [ctypes.POINTER(KVWindow), _c_int]),
                "txl_qkv_project": (_c_int, [_c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_int,
                                             _c_p, _c_p, ctypes.POINTER(KVWindow), _c_p,
                                             ctypes.POINTER(MemState), _c_p]),
                "txl_relattn_bwd_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
                "txl_relattn_bwd": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p,
                                             _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int,
                                             _c_int, _c_int, _c_int, _c_float, _c_int, _c_p,
                                             _c_size, _c_p]),
                "txl_relattn_fwd_noalloc": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_int, _c_p, _c_p,
                                                     _c_p, _c_p, _c_int, _c_int, _c_int, _c_int,
                                                     _c_int, _c_float, _c_int, _c_int, _c_p]),
                "txl_mem_concat": (_c_int, [_c_p, _c_p, ctypes.POINTER(MemState), _c_p, _c_int,
                                            _c_int, _c_int, _c_int, _c_p]),
                "txl_mem_update": (_c_int, [_c_p, ctypes.POINTER(MemState), _c_p, _c_int, _c_int,
                                            _c_int, _c_int, _c_p]),
                "txl_device_status": (_c_int, [_c_p]),
                "txl_set_wait_limit_ns": (_c_u64, [_c_u64]),
                "txl_debug_wait_timeout": (_c_int, [_c_u64, _c_p]),
                "txl_debug_checks": (_c_int, []),
                "txl_debug_index_probe": (_c_int, [_c_p]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().txl_status_string(int(status)).decode()


def version() -> int:
    return int(lib().txl_version())


def _check(rc: int, what: str):
    if rc != 0:
        raise TxlError(rc, f"{what}: {status_string(rc)} ({rc})")


def _stream(t: torch.Tensor | None = None, stream=None):
    if stream is None:
        dev = t.device if t is not None else torch.device("cuda", torch.cuda.current_device())
        stream = torch.cuda.current_stream(dev)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library takes device pointers)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return F32
    if dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"unsupported dtype {dtype} (float32 or bfloat16)")


def rel_pos_emb(K: int, d_model: int, dtype=torch.float32, device=None, out=None, stream=None):
    """Sinusoid relative table R [K, d_model]; row rho holds distance K-1-rho."""
    if out is None:
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        out = torch.empty(K, d_model, dtype=dtype, device=dev)
    _check(lib().txl_rel_pos_emb(_dev(out, "R"), int(K), int(d_model), _code(out.dtype),
                                 _stream(out, stream)), "txl_rel_pos_emb")
    return out


def workspace_size(B: int, H: int, L: int, dh: int, n_splits: int) -> int:
    return int(lib().txl_relattn_workspace_size(int(B), int(H), int(L), int(dh), int(n_splits)))


KERNELS = {1: "tc", 2: "decode", 3: "f32", 4: "decode_mma"}


def relattn_plan(B: int, H: int, M: int, L: int, dtype=torch.bfloat16, *, r_rows: int | None = None,
                 dh: int = 64, n_splits: int = 0, workspace_bytes: int = 0):
    """(kernel, splits) that relattn_fwd would use for these sizes: kernel is
    "tc", "decode" (one query, CUDA cores), "decode_mma" (2 to 8 queries,
    warp MMAs) or "f32".  Raises TxlError for sizes the call would reject."""
    kernel, splits = _c_int(0), _c_int(0)
    _check(lib().txl_relattn_plan(int(B), int(H), int(M), int(L),
                                  int(r_rows if r_rows is not None else M + L), int(dh),
                                  _code(dtype), int(n_splits), int(workspace_bytes),
                                  ctypes.byref(kernel), ctypes.byref(splits)), "txl_relattn_plan")
    return KERNELS[kernel.value], splits.value


def _kv_plane_stride(k, v):
    """0 for dense k, v; else the element stride between (b, h) planes when k and
    v are windows [B, H, K, dh] of larger buffers (rows contiguous within a plane,
    planes equally spaced)."""
    if k.is_contiguous() and v.is_contiguous():
        return 0
    B, H, K, dh = k.shape
    for t, name in ((k, "k"), (v, "v")):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the library takes device pointers)")
        st = t.stride()
        if st[3] != 1 or st[2] != dh or st[0] != H * st[1]:
            raise ValueError(f"{name}: rows of a plane must be contiguous and planes equally "
                             f"spaced (strides {st})")
    if k.stride() != v.stride():
        raise ValueError("k and v must have the same strides")
    return int(k.stride(1))


def relattn_fwd(q, k, v, r, u, v_bias, M: int, scale: float, *, out=None, lse=None,
                n_splits: int = 0, workspace=None, stream=None):
    """Relative-position attention of one layer.

    q [B,H,L,dh]; k, v [B,H,M+L,dh] (memory rows first); r [H,r_rows,dh] in the
    reversed order (row rho = W_kR R_{r_rows-1-rho}); u, v_bias [H,dh].  All
    bf16 (tensor-core path) or all fp32 (CUDA-core path).  k and v may be
    windows of larger buffers (e.g. ``kv_window_view``): rows contiguous, the
    (b, h) planes equally spaced; they then go through txl_relattn_fwd_strided.
    ``lse``: True to return log-sum-exp [B,H,L] (fp32), or a tensor to fill.
    Returns ``out`` or ``(out, lse)``."""
    B, H, L, dh = q.shape
    dt = q.dtype
    code = _code(dt)
    if out is None:
        out = torch.empty_like(q)
    want_lse = lse is not None and lse is not False
    if lse is True:
        lse = torch.empty(B, H, L, dtype=torch.float32, device=q.device)
    lse_ptr = _dev(lse, "lse", torch.float32) if want_lse else None
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    kv_stride = _kv_plane_stride(k, v)
    if kv_stride == 0:
        rc = lib().txl_relattn_fwd(
            _dev(q, "q", dt), _dev(k, "k", dt), _dev(v, "v", dt), _dev(r, "r", dt),
            int(r.shape[1]), _dev(u, "u", dt), _dev(v_bias, "v_bias", dt), _dev(out, "out", dt),
            lse_ptr, int(B), int(H), int(M), int(L), int(dh), float(scale), code, int(n_splits),
            ws_ptr, int(ws_bytes), _stream(q, stream))
        _check(rc, "txl_relattn_fwd")
    else:
        if k.dtype != dt or v.dtype != dt:
            raise ValueError(f"k and v must be {dt}")
        rc = lib().txl_relattn_fwd_strided(
            _dev(q, "q", dt), k.data_ptr(), v.data_ptr(), kv_stride, _dev(r, "r", dt),
            int(r.shape[1]), _dev(u, "u", dt), _dev(v_bias, "v_bias", dt), _dev(out, "out", dt),
            lse_ptr, int(B), int(H), int(M), int(L), int(dh), float(scale), code, int(n_splits),
            ws_ptr, int(ws_bytes), _stream(q, stream))
        _check(rc, "txl_relattn_fwd_strided")
    return (out, lse) if want_lse else out


def bwd_workspace_size(B: int, H: int, L: int, M: int) -> int:
    """Bytes of device workspace txl_relattn_bwd needs for a segment of L rows
    after a memory of M."""
    return int(lib().txl_relattn_bwd_workspace_size(int(B), int(H), int(L), int(M)))


def relattn_bwd(q, k, v, r, u, v_bias, dout, M: int, scale: float, *, grads=None,
                workspace=None, stream=None):
    """Backward of :func:`relattn_fwd` (bf16 inputs, same layouts) for the
    output gradient ``dout`` [B,H,L,dh].  Returns fp32
    ``(dq, dk, dv, dr, du, dv_bias)`` shaped like q, k, v, r, u, v_bias; dr, du,
    dv_bias are summed over the batch.  ``grads``: a tuple of such tensors to
    fill instead; ``workspace``: a device buffer of at least
    :func:`bwd_workspace_size` bytes (allocated when omitted)."""
    B, H, L, dh = q.shape
    bf = torch.bfloat16
    if grads is None:
        f = lambda t: torch.empty(t.shape, dtype=torch.float32, device=t.device)
        grads = (f(q), f(k), f(v), f(r), f(u), f(v_bias))
    dq, dk, dv, dr, du, dvb = grads
    if workspace is None:
        workspace = torch.empty(max(bwd_workspace_size(B, H, L, M), 256), dtype=torch.uint8,
                                device=q.device)
    f32 = torch.float32
    rc = lib().txl_relattn_bwd(
        _dev(q, "q", bf), _dev(k, "k", bf), _dev(v, "v", bf), _dev(r, "r", bf), int(r.shape[1]),
        _dev(u, "u", bf), _dev(v_bias, "v_bias", bf), _dev(dout, "dout", bf),
        _dev(dq, "dq", f32), _dev(dk, "dk", f32), _dev(dv, "dv", f32), _dev(dr, "dr", f32),
        _dev(du, "du", f32), _dev(dvb, "dv_bias", f32), int(B), int(H), int(M), int(L), int(dh),
        float(scale), BF16, _dev(workspace, "workspace"),
        int(workspace.numel() * workspace.element_size()), _stream(q, stream))
    _check(rc, "txl_relattn_bwd")
    return grads


def relattn_fwd_noalloc(q, k, v, r, u, v_bias, M: int, scale: float, *, out=None, lse=None,
                        n_splits: int = 0, stream=None):
    """relattn_fwd for callers that cannot allocate device memory at call time:
    split-key partial results go to the library's own scratch array (shared by
    all calls; calls that overlap on the GPU race on it).  The C entry point
    allocates nothing; a caller that cannot allocate passes ``out`` (and
    ``lse``) in, otherwise this wrapper creates them."""
    B, H, L, dh = q.shape
    dt = q.dtype
    code = _code(dt)
    if out is None:
        out = torch.empty_like(q)
    want_lse = lse is not None and lse is not False
    if lse is True:
        lse = torch.empty(B, H, L, dtype=torch.float32, device=q.device)
    lse_ptr = _dev(lse, "lse", torch.float32) if want_lse else None
    rc = lib().txl_relattn_fwd_noalloc(
        _dev(q, "q", dt), _dev(k, "k", dt), _dev(v, "v", dt), _dev(r, "r", dt), int(r.shape[1]),
        _dev(u, "u", dt), _dev(v_bias, "v_bias", dt), _dev(out, "out", dt), lse_ptr,
        int(B), int(H), int(M), int(L), int(dh), float(scale), code, int(n_splits),
        _stream(q, stream))
    _check(rc, "txl_relattn_fwd_noalloc")
    return (out, lse) if want_lse else out


def mem_concat(mem, state: MemState, h_new, out=None, stream=None):
    """Extended context [memory (oldest first) ; h_new] as [B, fill+L, d]."""
    B, L, d = h_new.shape
    if out is None:
        out = torch.empty(B, state.fill + L, d, dtype=h_new.dtype, device=h_new.device)
    mem_ptr = _dev(mem, "mem", h_new.dtype) if mem is not None and mem.numel() else None
    h_ptr = _dev(h_new, "h_new") if h_new.numel() else None
    ext_ptr = _dev(out, "ext", h_new.dtype) if out.numel() else None
    _check(lib().txl_mem_concat(ext_ptr, mem_ptr, ctypes.byref(state), h_ptr, int(B), int(L),
                                int(d), _code(h_new.dtype), _stream(h_new, stream)),
           "txl_mem_concat")
    return out


def mem_update(mem, state: MemState, h_new, stream=None):
    """Append h_new [B, L, d] to the ring-buffer memory mem [B, capacity, d];
    advances ``state`` in place."""
    B, L, d = h_new.shape
    mem_ptr = _dev(mem, "mem", h_new.dtype) if mem is not None and mem.numel() else None
    h_ptr = _dev(h_new, "h_new") if h_new.numel() else None
    _check(lib().txl_mem_update(mem_ptr, ctypes.byref(state), h_ptr, int(B),
                                int(L), int(d), _code(h_new.dtype), _stream(h_new, stream)),
           "txl_mem_update")
    return state


def kv_window_append(buf, state: KVWindow, seg, stream=None):
    """Append seg [planes, L, d] behind the memory rows of the window kept in buf
    [planes, capacity, d] (moving the memory to the buffer's front first when the
    rows would not fit); updates ``state.start`` in place."""
    P, L, d = seg.shape
    if buf.shape[0] != P or buf.shape[2] != d or buf.shape[1] != state.capacity:
        raise ValueError("buf must be [planes, capacity, d] matching seg and the state")
    _check(lib().txl_kv_window_append(_dev(buf, "buf", seg.dtype), ctypes.byref(state),
                                      _dev(seg, "seg") if seg.numel() else None, int(P), int(L),
                                      int(d), _code(seg.dtype), _stream(seg, stream)),
           "txl_kv_window_append")
    return state


def qkv_project(h, w, kv_buf, state: KVWindow, q=None, mem=None, mem_state: MemState | None = None,
                stream=None):
    """One layer's projections of the segment h [B, L, d_model] (bf16) by the
    stacked weights w [n_out*H*64, d_model] (W_q, W_kE, W_v rows when q is given,
    else W_kE, W_v): q into q [B, H, L, 64], k and v into the window rows behind
    the memory of kv_buf [2*B*H, capacity, 64] (keys' planes, then values'),
    and, when mem is given, h into the memory ring mem [B, capacity, d_model].
    Updates ``state.start`` and ``mem_state`` in place, as kv_window_append and
    mem_update do."""
    B, L, d = h.shape
    n_out = 3 if q is not None else 2
    if w.shape[1] != d or w.shape[0] % (n_out * 64):
        raise ValueError("w must be [n_out * H * 64, d_model]")
    H = w.shape[0] // (n_out * 64)
    if kv_buf.shape != (2 * B * H, state.capacity, 64):
        raise ValueError("kv_buf must be [2 * B * H, capacity, 64]")
    if q is not None and tuple(q.shape) != (B, H, L, 64):
        raise ValueError("q must be [B, H, L, 64]")
    if (mem is None) != (mem_state is None):
        raise ValueError("mem and mem_state go together")
    _check(lib().txl_qkv_project(_dev(h, "h", torch.bfloat16), _dev(w, "w", torch.bfloat16),
                                 int(B), int(L), int(d), int(H), 64,
                                 _dev(q, "q", torch.bfloat16) if q is not None else None,
                                 _dev(kv_buf, "kv_buf", torch.bfloat16), ctypes.byref(state),
                                 _dev(mem, "mem", torch.bfloat16) if mem is not None else None,
                                 ctypes.byref(mem_state) if mem_state is not None else None,
                                 _stream(h, stream)),
           "txl_qkv_project")
    return state


def kv_window_advance(state: KVWindow, L: int):
    """After attending to the appended segment of L rows: keep the newest M rows."""
    _check(lib().txl_kv_window_advance(ctypes.byref(state), int(L)), "txl_kv_window_advance")
    return state


def kv_window_view(buf, state: KVWindow, L: int, B: int, H: int):
    """The window [memory ; segment] of buf [B*H, capacity, d] as a [B, H, fill+L, d]
    view (no copy), for relattn_fwd."""
    d = buf.shape[2]
    return buf.view(B, H, state.capacity, d)[:, :, state.start:state.start + state.fill + L]


def device_status(stream=None) -> int:
    """Synchronise and return (and clear) the kernels' device status word."""
    return int(lib().txl_device_status(_stream(None, stream)))


def set_wait_limit_ns(ns: int) -> int:
    return int(lib().txl_set_wait_limit_ns(int(ns)))


def debug_wait_timeout(ns: int, stream=None) -> int:
    return int(lib().txl_debug_wait_timeout(int(ns), _stream(None, stream)))


def debug_checks() -> bool:
    """True when the loaded library is the debug build (device-side index checks)."""
    return bool(lib().txl_debug_checks())


def debug_index_probe(stream=None) -> int:
    """Fail one device-side index check on purpose; returns the status then read
    (TXL_ERR_INDEX = -8 in the debug build, 0 in a release build)."""
    return int(lib().txl_debug_index_probe(_stream(None, stream)))
