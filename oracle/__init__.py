"""fp64 CPU oracle for diagonal-decay gated linear attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this package.  The CUDA library never imports, links or
calls it, and it shares no code with the library.

* ``gla_fwd`` / ``gla_bwd`` wrap the plain C token recurrence and its
  brute-force adjoint in ``oracle.c`` (fp64, pthreads).
* ``chunked.py`` holds the segmented/chunked fp64 form written from the ZeCO
  pages, used only to pin the recurrence against the pages' decomposition.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(hand-worked cases, the alpha=1 causal-attention special case, a closed form,
the chunked form, central finite differences, and the dlog_alpha identity),
and planted mistakes in copies of oracle.c are each caught by those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into oracle/_build/liboracle.so (portable flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", "-pthread", _SRC,
               "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


def configure(lib):
    """Declare the argument types of a loaded oracle library and return it."""
    i64, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.oracle_gla_fwd.argtypes = [i64] * 5 + [dp] * 5 + [i64, ip, dp, dp, ctypes.c_int]
    lib.oracle_gla_fwd.restype = ctypes.c_int
    lib.oracle_gla_bwd.argtypes = ([i64] * 5 + [dp] * 7 + [i64, ip, dp, dp, dp, dp] +
                                   [i64, ip, dp, ctypes.c_int])
    lib.oracle_gla_bwd.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = configure(ctypes.CDLL(build()))
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _idx(ix):
    if ix is None:
        return None
    return np.ascontiguousarray(np.asarray(ix, dtype=np.int64))


def gla_fwd(q, k, v, log_alpha, S0=None, cols=None, nthreads=None):
    """Token-recurrence forward in fp64.

    Returns ``(o, S_final)`` with ``o`` [B,H,T,ncols] and ``S_final``
    [B,H,dk,ncols]; ``cols`` selects d_v columns (None: all).
    """
    q, k, v, g, S0 = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(S0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape == g.shape and v.shape == (B, H, T, dv)
    if S0 is not None:
        assert S0.shape == (B, H, dk, dv)
    cols = _idx(cols)
    nc = dv if cols is None else len(cols)
    o = np.zeros((B, H, T, nc))
    sf = np.zeros((B, H, dk, nc))
    rc = _load().oracle_gla_fwd(B, H, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S0),
                                nc, _ptr(cols), _ptr(o), _ptr(sf),
                                nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_gla_fwd failed ({rc})")
    return o, sf


def gla_bwd(q, k, v, log_alpha, S0, do, dS_final, rows=None, cols=None, nthreads=None,
            want_rows=True, want_cols=True):
    """Brute-force adjoint in fp64.

    Returns a dict: ``dq``, ``dk``, ``dlog_alpha`` [B,H,T,nrows], ``dS0``
    [B,H,nrows,dv] for the selected d_k rows, and ``dv`` [B,H,T,ncols] for the
    selected d_v columns (None: all rows / all columns).
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(log_alpha)
    S0, do, dSf = _f64(S0), _f64(do), _f64(dS_final)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    rows, cols = _idx(rows), _idx(cols)
    nr = (dk if rows is None else len(rows)) if want_rows else 0
    nc = (dv if cols is None else len(cols)) if want_cols else 0
    dq = np.zeros((B, H, T, nr))
    dk_ = np.zeros((B, H, T, nr))
    dg = np.zeros((B, H, T, nr))
    dS0 = np.zeros((B, H, nr, dv))
    dv_ = np.zeros((B, H, T, nc))
    rc = _load().oracle_gla_bwd(B, H, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(S0),
                                _ptr(do), _ptr(dSf), nr, _ptr(rows), _ptr(dq), _ptr(dk_),
                                _ptr(dg), _ptr(dS0), nc, _ptr(cols), _ptr(dv_),
                                nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_gla_bwd failed ({rc})")
    return dict(dq=dq, dk=dk_, dlog_alpha=dg, dS0=dS0, dv=dv_)


def boundary_states(q, k, v, log_alpha, S0, P, nthreads=None):
    """States entering each segment: S_in[p] = state after token p*L-1 (S_in[0] = S0).

    Returns [B,H,P+1,dk,dv]; S_in[P] is S_final.  Computed with the plain
    recurrence on prefixes, so it is independent of any chunked evaluation.
    """
    q, k, v, g, S0 = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(S0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    L = T // P
    out = np.zeros((B, H, P + 1, dk, dv))
    out[:, :, 0] = 0.0 if S0 is None else S0
    S = S0
    for p in range(P):
        sl = slice(p * L, (p + 1) * L)
        _, S = gla_fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], g[:, :, sl], S,
                       nthreads=nthreads)
        out[:, :, p + 1] = S
    return out


def boundary_states_cols(q, k, v, log_alpha, S0, P, cols, nthreads=None):
    """Columns ``cols`` of the segment-entry states S_in[p], p = 0..P (fp64).

    Every column of the state evolves on its own (the decay scales rows), so the
    selected columns can be carried from prefix to prefix without the others.
    Returns [B,H,P+1,dk,ncols].
    """
    q, k, v, g, S0 = _f64(q), _f64(k), _f64(v), _f64(log_alpha), _f64(S0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    cols = _idx(cols)
    L = T // P
    S = np.zeros((B, H, dk, dv)) if S0 is None else S0.copy()
    out = np.zeros((B, H, P + 1, dk, len(cols)))
    out[:, :, 0] = S[..., cols]
    for p in range(P):
        sl = slice(p * L, (p + 1) * L)
        _, sf = gla_fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], g[:, :, sl], S, cols=cols,
                        nthreads=nthreads)
        S[..., cols] = sf
        out[:, :, p + 1] = sf
    return out


# ---- other decay forms.  The ZeCO pages leave linear attention with other
# decays to future work (ZeCO: Limitations); the LASP page's linear attention
# has none.  A per-token scalar decay multiplies every d_k row of the state by
# the same alpha_t (RetNet / Lightning-style); "none" is alpha = 1.  Both are the
# diagonal recurrence with log_alpha[t, i] = g_t (resp. 0), and the gradient
# with respect to a scalar g_t is the sum over i of the diagonal one (chain
# rule through the broadcast).  Pinned by a closed form (constant scalar
# decay = causal attention weighted by e^{c (t - s)}), by the alpha = 1 causal
# form and by central finite differences with respect to the scalar g.

DECAY_DIAG, DECAY_SCALAR, DECAY_NONE = 0, 1, 2


def expand_log_alpha(log_alpha, decay, shape):
    """The [B,H,T,dk] log-decay of a decay form (log_alpha [B,H,T] when scalar,
    ignored when none)."""
    if decay == DECAY_DIAG:
        return _f64(log_alpha)
    B, H, T, dk = shape
    if decay == DECAY_SCALAR:
        return np.ascontiguousarray(np.broadcast_to(_f64(log_alpha)[..., None], (B, H, T, dk)))
    return np.zeros((B, H, T, dk))


def gla_fwd_decay(q, k, v, log_alpha, S0, decay, cols=None, nthreads=None):
    """Forward of a decay form: (o, S_final)."""
    return gla_fwd(q, k, v, expand_log_alpha(log_alpha, decay, q.shape), S0, cols, nthreads)


def gla_bwd_decay(q, k, v, log_alpha, S0, do, dS_final, decay, nthreads=None):
    """Backward of a decay form: dlog_alpha is [B,H,T] for a scalar decay and
    None without decay."""
    r = gla_bwd(q, k, v, expand_log_alpha(log_alpha, decay, q.shape), S0, do, dS_final,
                nthreads=nthreads)
    if decay == DECAY_SCALAR:
        r["dlog_alpha"] = r["dlog_alpha"].sum(axis=-1)
    elif decay == DECAY_NONE:
        r["dlog_alpha"] = None
    return r
