"""Segmented (ZeCO-style) gated linear attention on one GB300 -- Python binding.

This module only marshals arguments: it allocates outputs with PyTorch on the
current CUDA device and calls the C ABI of libzeco_gla.so (declared in
include/zeco_gla.h) on the current stream.  Every step of the computation runs
in the library's CUDA kernels.  There is no CPU or PyTorch fallback: if the
library is not built, or no GPU is present, the calls raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libzeco_gla.so")

ZECO_OK, ZECO_ERR_ARG, ZECO_ERR_UNSUPPORTED, ZECO_ERR_WORKSPACE, ZECO_ERR_CUDA = 0, -1, -2, -3, -4
ZECO_ERR_TIMEOUT = -5
OVERLAP_DEFAULT = 4  # ZECO_OVERLAP_DEFAULT
ZECO_F32, ZECO_BF16 = 0, 1
PATH_AUTO, PATH_SIMT, PATH_TC = 0, 1, 2
_PATHS = {"auto": PATH_AUTO, "simt": PATH_SIMT, "tc": PATH_TC}

EXPORTED = ["zeco_gla_saved_bytes", "zeco_gla_workspace_bytes", "zeco_gla_fwd", "zeco_gla_bwd",
            "zeco_strerror", "zeco_gla_resolve_path", "zeco_gla_segments",
            "zeco_check_device_status", "zeco_last_device_status", "zeco_selftest_bounded_wait",
            "zeco_set_profile_events", "zeco_profile_event_count", "zeco_profile_kernel_name",
            "zeco_set_overlap", "zeco_gla_bwd_noalloc"]


class ZecoShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("T", ctypes.c_int64),
                ("dk", ctypes.c_int64), ("dv", ctypes.c_int64), ("P", ctypes.c_int32),
                ("K", ctypes.c_int32), ("C", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("path", ctypes.c_int32), ("decay", ctypes.c_int32)]


class ZecoError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (code {code})")
        self.code = code


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libzeco_gla.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library not built: {path} is missing "
                    "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
            lib = ctypes.CDLL(path)
            vp, sz, sp = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ZecoShape)
            lib.zeco_gla_saved_bytes.argtypes = [sp]
            lib.zeco_gla_saved_bytes.restype = sz
            lib.zeco_gla_segments.argtypes = [sp]
            lib.zeco_gla_segments.restype = ctypes.c_int64
            lib.zeco_set_overlap.argtypes = [ctypes.c_int]
            lib.zeco_set_overlap.restype = ctypes.c_int
            lib.zeco_gla_workspace_bytes.argtypes = [sp, ctypes.c_int]
            lib.zeco_gla_workspace_bytes.restype = sz
            lib.zeco_gla_fwd.argtypes = [sp] + [vp] * 8 + [vp, sz, vp]
            lib.zeco_gla_fwd.restype = ctypes.c_int
            lib.zeco_gla_bwd.argtypes = [sp] + [vp] * 12 + [vp, sz, vp]
            lib.zeco_gla_bwd.restype = ctypes.c_int
            lib.zeco_strerror.argtypes = [ctypes.c_int]
            lib.zeco_strerror.restype = ctypes.c_char_p
            lib.zeco_gla_resolve_path.argtypes = [sp]
            lib.zeco_gla_resolve_path.restype = ctypes.c_int
            lib.zeco_selftest_bounded_wait.argtypes = [vp]
            lib.zeco_selftest_bounded_wait.restype = ctypes.c_int
            lib.zeco_check_device_status.argtypes = []
            lib.zeco_check_device_status.restype = ctypes.c_int
            lib.zeco_last_device_status.argtypes = [vp]
            lib.zeco_last_device_status.restype = ctypes.c_int
            lib.zeco_gla_bwd_noalloc.argtypes = [sp] + [vp] * 13
            lib.zeco_gla_bwd_noalloc.restype = ctypes.c_int
            _lib = lib
    return _lib


# decay forms: per d_k row (gated linear attention), one per token, none
DECAY_DIAG, DECAY_SCALAR, DECAY_NONE = 0, 1, 2
_DECAYS = {"diag": DECAY_DIAG, "scalar": DECAY_SCALAR, "none": DECAY_NONE}


def make_shape(B, H, T, dk, dv, P, K, C, dtype, path="auto", decay="diag") -> ZecoShape:
    if isinstance(dtype, torch.dtype):
        dt = ZECO_BF16 if dtype == torch.bfloat16 else ZECO_F32
    else:
        dt = ZECO_BF16 if dtype in ("bf16", ZECO_BF16) else ZECO_F32
    return ZecoShape(B, H, T, dk, dv, P, K, C, dt, _PATHS.get(path, path),
                     _DECAYS.get(decay, decay))


def _check(rc):
    if rc != ZECO_OK:
        raise ZecoError(rc, load_library().zeco_strerror(rc).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def saved_bytes(shape: ZecoShape) -> int:
    return load_library().zeco_gla_saved_bytes(ctypes.byref(shape))


def workspace_bytes(shape: ZecoShape, bwd: bool) -> int:
    return load_library().zeco_gla_workspace_bytes(ctypes.byref(shape), int(bwd))


def segments(shape: ZecoShape) -> int:
    """Segments the library evaluates for this shape (P, or P split further when
    B*H*P is too small to fill the GPU); the `saved` layout follows it."""
    n = load_library().zeco_gla_segments(ctypes.byref(shape))
    if n < 0:
        _check(int(n))
    return int(n)


def check_device_status() -> None:
    """Raise ZecoError if a bounded device wait gave up since the last check
    (synchronise the streams of the calls to cover first).  The flags are per
    device: a give-up on any stream of the current device is reported."""
    _check(load_library().zeco_check_device_status())


def last_device_status(stream=None) -> int:
    """zeco_last_device_status: synchronise ``stream`` (default: the current
    stream), then read and clear the device's bounded-wait flags.  Returns the
    code (ZECO_OK or ZECO_ERR_TIMEOUT, ZECO_ERR_CUDA) without raising."""
    return int(load_library().zeco_last_device_status(_stream_ptr(stream)))


def selftest_bounded_wait(stream=None) -> None:
    """Launch the library's diagnostic kernel, four warps whose waits can never
    complete (the first gives up after 2 s, the others then at once; it records
    ZECO_ERR_TIMEOUT for check_device_status)."""
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(load_library().zeco_selftest_bounded_wait(ctypes.c_void_p(st.cuda_stream)))


def set_overlap(mode: int) -> None:
    """Schedule of the work beside the segment scan: 1 the scan-independent score
    passes on a second stream, 2 the segment scan on a second stream beside them
    (the pages' schedule), 3 (forward) pass 2 per block of segments as soon as the
    scan reaches it, 4 (OVERLAP_DEFAULT) mode 1 plus the dq/dk sweeps on a
    high-priority stream beside the dv sweep, 0 everything on one stream."""
    _check(load_library().zeco_set_overlap(int(mode)))


def resolve_path(shape: ZecoShape) -> str:
    rc = load_library().zeco_gla_resolve_path(ctypes.byref(shape))
    if rc < 0:
        _check(rc)
    return {PATH_SIMT: "simt", PATH_TC: "tc"}[rc]


def _on(stream):
    """Allocate on the stream the kernels run on, so the caching allocator
    orders reuse of these blocks after the launches that use them."""
    if isinstance(stream, torch.cuda.Stream):
        return torch.cuda.stream(stream)
    return contextlib.nullcontext()


def _shape_of(q, v, P, K, C, path, decay="diag"):
    B, H, T, dk = q.shape
    return make_shape(B, H, T, dk, v.shape[-1], P, K, C, q.dtype, path, decay)


def _expect(t, name, device, shape=None, dtype=None, nbytes=None, optional=True):
    """Raise ValueError unless ``t`` is a contiguous tensor on ``device`` with the
    given shape and dtype (and at least ``nbytes`` bytes).  The library reads and
    writes these buffers through raw pointers, so nothing else is safe to pass."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name}: a tensor is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if nbytes is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name}: {t.numel() * t.element_size()} bytes, needs {nbytes}")


def _check_inputs(q, k, v, log_alpha, decay):
    """The inputs of both directions: q, k [B,H,T,dk] and v [B,H,T,dv] of one I/O dtype
    (fp32 or bf16) on one CUDA device; log_alpha in the layout of the decay form."""
    if not isinstance(q, torch.Tensor) or q.dim() != 4:
        raise ValueError("q: expected a [B, H, T, dk] tensor")
    if q.device.type != "cuda":
        raise ValueError(f"q: on {q.device}; the library runs on CUDA devices only")
    if q.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"q: dtype {q.dtype}; fp32 and bf16 are supported")
    B, H, T, dk = q.shape
    _expect(q, "q", q.device)
    _expect(k, "k", q.device, q.shape, q.dtype, optional=False)
    if not isinstance(v, torch.Tensor) or v.dim() != 4 or tuple(v.shape[:3]) != (B, H, T):
        raise ValueError("v: expected a [B, H, T, dv] tensor matching q")
    _expect(v, "v", q.device, None, q.dtype)
    if decay != "none" and _DECAYS.get(decay, decay) != DECAY_NONE:
        g_shape = (B, H, T) if _DECAYS.get(decay, decay) == DECAY_SCALAR else (B, H, T, dk)
        _expect(log_alpha, "log_alpha", q.device, g_shape, q.dtype, optional=False)
    return (B, H, dk, v.shape[-1])


def zeco_gla_fwd(q, k, v, log_alpha, S0=None, *, P, K, C, path="auto", o=None, S_final=None,
                 saved=None, workspace=None, stream=None, want_S_final=True, decay="diag"):
    """Forward through the C ABI.  Returns (o, S_final or None, saved).

    q, k: [B,H,T,dk]; v: [B,H,T,dv] (fp32 or bf16, CUDA, contiguous); log_alpha:
    [B,H,T,dk] (decay "diag"), [B,H,T] ("scalar") or None ("none").
    S0: [B,H,dk,dv] fp32 or None (zeros).  ``saved`` must be passed to the backward
    with the same P, K, C, path and decay: its layout follows the resolved path (on the
    tensor-core path it also keeps the forward's decay-weighted operands and masked
    scores, which the backward reads instead of recomputing).
    ``workspace``: a uint8 buffer of at least workspace_bytes(shape, False) bytes,
    allocated here when None.
    """
    B, H, dk, dv = _check_inputs(q, k, v, log_alpha, decay)
    dev = q.device
    state = (B, H, dk, dv)
    _expect(S0, "S0", dev, state, torch.float32)
    _expect(o, "o", dev, v.shape, v.dtype)
    _expect(S_final, "S_final", dev, state, torch.float32)
    shape = _shape_of(q, v, P, K, C, path, decay)
    nsaved = saved_bytes(shape)  # 0 for a shape the library rejects (it says why below)
    _expect(saved, "saved", dev, nbytes=nsaved)
    nws = workspace_bytes(shape, False)
    _expect(workspace, "workspace", dev, nbytes=nws)
    with _on(stream):
        if o is None:
            o = torch.empty(v.shape, dtype=v.dtype, device=dev)
        if want_S_final and S_final is None:
            S_final = torch.empty(q.shape[0], q.shape[1], q.shape[-1], v.shape[-1],
                                  dtype=torch.float32, device=dev)
        if saved is None:
            saved = torch.empty(max(saved_bytes(shape), 16), dtype=torch.uint8, device=dev)
        if workspace is None and nws:
            workspace = torch.empty(nws, dtype=torch.uint8, device=dev)
    ws_len = workspace.numel() if workspace is not None else 0
    rc = load_library().zeco_gla_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(log_alpha), _ptr(S0), _ptr(o), _ptr(S_final),
                                     _ptr(saved), _ptr(workspace), ws_len, _stream_ptr(stream))
    _check(rc)
    return o, S_final, saved


def zeco_gla_bwd(q, k, v, log_alpha, saved, do, dS_final=None, *, P, K, C, path="auto",
                 grads=None, workspace=None, stream=None, want_dS0=True, decay="diag"):
    """Backward through the C ABI.  Returns dict(dq, dk, dv, dlog_alpha, dS0);
    dlog_alpha has log_alpha's shape and is None without decay."""
    B, H, dk, dv = _check_inputs(q, k, v, log_alpha, decay)
    dev = q.device
    state = (B, H, dk, dv)
    shape = _shape_of(q, v, P, K, C, path, decay)
    _expect(saved, "saved", dev, nbytes=saved_bytes(shape), optional=False)
    _expect(do, "do", dev, v.shape, v.dtype, optional=False)
    _expect(dS_final, "dS_final", dev, state, torch.float32)
    if grads is not None:
        _expect(grads.get("dq"), "dq", dev, q.shape, q.dtype, optional=False)
        _expect(grads.get("dk"), "dk", dev, k.shape, k.dtype, optional=False)
        _expect(grads.get("dv"), "dv", dev, v.shape, v.dtype, optional=False)
        if log_alpha is not None:
            _expect(grads.get("dlog_alpha"), "dlog_alpha", dev, log_alpha.shape,
                    log_alpha.dtype, optional=False)
        _expect(grads.get("dS0"), "dS0", dev, state, torch.float32)
    nws = workspace_bytes(shape, True)
    _expect(workspace, "workspace", dev, nbytes=nws)
    with _on(stream):
        if grads is None:
            grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k),
                         dv=torch.empty_like(v),
                         dlog_alpha=None if log_alpha is None else torch.empty_like(log_alpha))
            if want_dS0:
                grads["dS0"] = torch.empty(q.shape[0], q.shape[1], q.shape[-1], v.shape[-1],
                                           dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    rc = load_library().zeco_gla_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(log_alpha), _ptr(saved), _ptr(do), _ptr(dS_final),
                                     _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]),
                                     _ptr(grads["dlog_alpha"]), _ptr(grads.get("dS0")),
                                     _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _check(rc)
    return grads
