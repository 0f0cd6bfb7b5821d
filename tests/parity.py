"""Helpers for the GPU parity tests: run the library, run the oracle, compare."""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import oracle

TOL_F32 = 1e-4  # max relative error (normwise infinity) for fp32 I/O
TOL_BF16 = 2e-2  # relative L2 error for bf16 I/O with fp32 accumulation


def max_rel(x, r) -> float:
    """max|x - r| / max|r| over the tensor (normwise infinity relative error)."""
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    den = np.abs(r).max() if r.size else 0.0
    return float(np.abs(x - r).max() / den) if den > 0 else float(np.abs(x - r).max())


def rel_l2(x, r) -> float:
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    den = np.linalg.norm(r)
    return float(np.linalg.norm(x - r) / den) if den > 0 else float(np.linalg.norm(x - r))


def err(x, r, dtype) -> float:
    return max_rel(x, r) if dtype == "f32" else rel_l2(x, r)


def tol(dtype) -> float:
    return TOL_F32 if dtype == "f32" else TOL_BF16


def to_np(t):
    return t.detach().float().cpu().numpy()


def run_gpu(z, x, P, K, C, path="auto", bwd=True, dev="cuda"):
    """Forward (+ backward) through the C ABI on device tensors."""
    g = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, sf, saved = z.zeco_gla_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["S0"], P=P, K=K,
                                  C=C, path=path)
    out = dict(o=o, S_final=sf, saved=saved)
    if bwd:
        out.update(z.zeco_gla_bwd(g["q"], g["k"], g["v"], g["log_alpha"], saved, g["do"],
                                  g["dS_final"], P=P, K=K, C=C, path=path))
    torch.cuda.synchronize()
    z.check_device_status()  # no bounded device wait gave up
    return out


def saved_states(saved, B, H, P, dk, dv):
    n = B * H * (P + 1) * dk * dv
    return saved.view(torch.float32)[:n].view(B, H, P + 1, dk, dv)


def compare_full(z, x, P, K, C, dtype, path="auto", bwd=True, check_states=True):
    """Full-tensor parity of every output against the oracle; returns the errors."""
    res = run_gpu(z, x, P, K, C, path=path, bwd=bwd)
    B, H, T, dk = x["q"].shape
    dv = x["v"].shape[-1]
    ro, rsf = oracle.gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"])
    errs = {"o": err(to_np(res["o"]), ro, dtype), "S_final": err(to_np(res["S_final"]), rsf, dtype)}
    if check_states:
        # the library may split the P segments further (zeco_gla_segments)
        pe = z.segments(z.make_shape(B, H, T, dk, dv, P, K, C, dtype, path))
        assert pe % P == 0
        bs = oracle.boundary_states(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], pe)
        got = to_np(saved_states(res["saved"], B, H, pe, dk, dv))
        errs["S_in"] = err(got, bs, dtype)
    if bwd:
        rg = oracle.gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], x["do"],
                            x["dS_final"])
        for n in ("dq", "dk", "dv", "dlog_alpha", "dS0"):
            errs[n] = err(to_np(res[n]), rg[n], dtype)
    return errs


def kernel_names(z, run):
    """Run ``run()`` with the library's per-kernel profiling marks on and return
    (names of the kernels it launched, in launch order; run's result)."""
    lib = z.load_library()
    n = 64
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()  # materialise the handles
    torch.cuda.synchronize()
    handles = (ctypes.c_void_p * n)(*[e.cuda_event for e in evs])
    lib.zeco_set_profile_events.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.zeco_profile_kernel_name.restype = ctypes.c_char_p
    lib.zeco_set_profile_events(ctypes.cast(handles, ctypes.c_void_p), n)
    try:
        out = run()
        cnt = lib.zeco_profile_event_count()
        names = [lib.zeco_profile_kernel_name(i).decode() for i in range(cnt // 2)]
    finally:
        lib.zeco_set_profile_events(None, 0)
    torch.cuda.synchronize()
    return names, out


def chunk_rows(T, segments, C=64, first=2, last=2):
    """Token indices of the first ``first`` and last ``last`` chunks of every one
    of ``segments`` equal segments (where the carried states weigh most)."""
    L = T // segments
    idx = []
    for p in range(segments):
        a = p * L
        idx.extend(range(a, a + first * C))
        idx.extend(range(a + L - last * C, a + L))
    return np.unique(np.asarray(idx))
