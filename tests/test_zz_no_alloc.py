"""zeco_gla_bwd_noalloc: the backward for callers that cannot allocate.

Callers such as plugins inside a framework that owns all device memory, or
code running where cudaMalloc may not be called, cannot hand the backward a
workspace.  This entry point keeps its scratch in a fixed array inside the
library.  These tests call it through the C ABI and check that it returns
what zeco_gla_bwd returns, on two calls in a row (the array keeps the previous
call's contents, which must not leak into the next result), and that shapes
needing more scratch than the array holds are refused.

The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dlog_alpha", "dS0")


@pytest.fixture(scope="module")
def z():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_state_scan_gb300 import build
    build.build()
    import chunked_state_scan_gb300 as pkg
    lib = pkg.load_library()
    vp = ctypes.c_void_p
    lib.zeco_gla_bwd_noalloc.argtypes = [ctypes.POINTER(pkg.ZecoShape)] + [vp] * 13
    lib.zeco_gla_bwd_noalloc.restype = ctypes.c_int
    return pkg


def _noalloc_bwd(z, shape, x, saved, stream):
    out = {n: torch.full_like(x[n2], float("nan")) for n, n2 in
           (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dlog_alpha", "log_alpha"),
            ("dS0", "S0"))}
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = z.load_library().zeco_gla_bwd_noalloc(
        ctypes.byref(shape), p(x["q"]), p(x["k"]), p(x["v"]), p(x["log_alpha"]), p(saved),
        p(x["do"]), p(x["dS_final"]), p(out["dq"]), p(out["dk"]), p(out["dv"]),
        p(out["dlog_alpha"]), p(out["dS0"]), ctypes.c_void_p(stream.cuda_stream))
    return rc, out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_matches_workspace_backward_twice(z, dtype):
    w = workloads.TINY_F32.replace(dtype=dtype, s0_scale=0.2)
    x = {n: t.cuda() for n, t in workloads.make_inputs(w).items()}
    stream = torch.cuda.current_stream()
    shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, dtype)
    assert z.workspace_bytes(shape, True) <= 32 << 20
    _, _, saved = z.zeco_gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], P=w.P,
                                 K=w.K, C=w.C)
    ref = z.zeco_gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], saved, x["do"],
                         x["dS_final"], P=w.P, K=w.K, C=w.C)
    for call in range(2):
        # the second call sees a different upstream gradient, so stale scratch
        # from the first call would show up in its result
        xx = dict(x)
        if call == 1:
            xx["do"] = -2.0 * x["do"]
            xx["dS_final"] = -2.0 * x["dS_final"]
            ref = z.zeco_gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], saved, xx["do"],
                                 xx["dS_final"], P=w.P, K=w.K, C=w.C)
        rc, got = _noalloc_bwd(z, shape, xx, saved, stream)
        assert rc == 0, z.load_library().zeco_strerror(rc)
        torch.cuda.synchronize()
        for n in GRADS:
            e = parity.err(parity.to_np(got[n]), parity.to_np(ref[n]), dtype)
            assert e <= parity.tol(dtype), (call, n, e)


def test_noalloc_refuses_shapes_beyond_its_scratch(z):
    # the 1M-token workload needs ~5 GB of backward scratch, far above the array
    w = workloads.LONG_FWDBWD
    shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype)
    assert z.workspace_bytes(shape, True) > 32 << 20
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = z.load_library().zeco_gla_bwd_noalloc(ctypes.byref(shape), *([p] * 6), None,
                                               *([p] * 4), None, None)
    assert rc == z.ZECO_ERR_WORKSPACE
