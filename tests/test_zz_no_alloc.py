"""zeco_gla_bwd_noalloc: the backward for callers that cannot allocate.

Callers such as plugins inside a framework that owns all device memory, or
code running where cudaMalloc may not be called, cannot hand the backward a
workspace.  This entry point keeps its scratch in a fixed array inside the
library.  These tests call it through the C ABI and check that it returns
what zeco_gla_bwd returns, on two calls in a row.  The array keeps the
previous call's contents, which must not leak into the next result, so before
the checked calls the array is filled by a call on a different, larger shape,
and the second call sees a different upstream gradient.  Shapes needing more
scratch than the array holds are refused, and argument errors come back with
zeco_gla_bwd's codes.

The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dlog_alpha", "dS0")
MAX_WS = 32 << 20


@pytest.fixture(scope="module")
def z():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_state_scan_gb300 import build
    build.build()
    import chunked_state_scan_gb300 as pkg
    pkg.load_library()
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


def _fill_array_with_other_data(z, stream):
    """A valid call on a different, larger tensor-core shape (about 14 MB of
    scratch): it leaves the shared array full of unrelated values."""
    w = workloads.Workload("fill", B=1, H=2, T=4096, dk=128, dv=512, P=2, K=2, C=64,
                           dtype="bf16", seed=99, qk_scale=1 / 16, v_scale=1.0, x_mean=1.0,
                           s0_scale=0.3, bwd=True)
    shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype)
    need = z.workspace_bytes(shape, True)
    assert 8 << 20 < need <= MAX_WS
    x = {n: t.cuda() for n, t in workloads.make_inputs(w).items()}
    _, _, saved = z.zeco_gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], P=w.P,
                                 K=w.K, C=w.C)
    rc, _ = _noalloc_bwd(z, shape, x, saved, stream)
    assert rc == 0, z.load_library().zeco_strerror(rc)
    torch.cuda.synchronize()


# fp32 and bf16 on the CUDA-core path (d_k = 64; d_v = 64, and for bf16 d_v = 96,
# off the tensor-core kernels' 64-column grid), and a bf16 shape on the
# tensor-core path, whose backward also keeps the score gradient dA in the array
# and writes it from a second stream
CASES = {
    "f32_simt": (workloads.TINY_F32.replace(dtype="f32", s0_scale=0.2), "simt"),
    "bf16_simt": (workloads.TINY_F32.replace(dtype="bf16", s0_scale=0.2, dv=96), "simt"),
    "bf16_tc": (workloads.Workload("tc", B=1, H=1, T=2048, dk=128, dv=512, P=2, K=4, C=64,
                                   dtype="bf16", seed=12, qk_scale=1 / 16, v_scale=1.0,
                                   x_mean=0.0, s0_scale=0.2, bwd=True), "tc"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_workspace_backward_twice(z, case):
    w, path = CASES[case]
    x = {n: t.cuda() for n, t in workloads.make_inputs(w).items()}
    stream = torch.cuda.current_stream()
    shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype)
    assert z.resolve_path(shape) == path
    assert z.workspace_bytes(shape, True) <= MAX_WS
    _, _, saved = z.zeco_gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], P=w.P,
                                 K=w.K, C=w.C)
    _fill_array_with_other_data(z, stream)
    for call in range(2):
        # the second call sees a different upstream gradient, so stale scratch
        # from the first call would show up in its result
        xx = dict(x)
        if call == 1:
            xx["do"] = (-2.0 * x["do"].float()).to(x["do"].dtype)
            xx["dS_final"] = -2.0 * x["dS_final"]
        ref = z.zeco_gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], saved, xx["do"],
                             xx["dS_final"], P=w.P, K=w.K, C=w.C)
        rc, got = _noalloc_bwd(z, shape, xx, saved, stream)
        assert rc == 0, z.load_library().zeco_strerror(rc)
        torch.cuda.synchronize()
        assert z.last_device_status() == z.ZECO_OK
        for n in GRADS:
            e = parity.err(parity.to_np(got[n]), parity.to_np(ref[n]), w.dtype)
            assert e <= parity.tol(w.dtype), (case, call, n, e)


def test_noalloc_refuses_shapes_beyond_its_scratch(z):
    # the 1M-token workload needs ~5 GB of backward scratch, far above the array
    w = workloads.LONG_FWDBWD
    shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype)
    assert z.workspace_bytes(shape, True) > MAX_WS
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = z.load_library().zeco_gla_bwd_noalloc(ctypes.byref(shape), *([p] * 6), None,
                                               *([p] * 4), None, None)
    assert rc == z.ZECO_ERR_WORKSPACE


def test_noalloc_argument_errors_match_the_workspace_backward(z):
    # the same shape and pointer checks as zeco_gla_bwd, before the size check:
    # a null pointer on an oversized shape is an argument error, not a size error
    lib = z.load_library()
    dummy = torch.empty(64, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    ws = ctypes.c_void_p(dummy.data_ptr())
    big = z.make_shape(1, 4, 1 << 20, 256, 512, 64, 8, 64, "bf16")
    cases = [
        (big, [p] * 6 + [None] + [None] + [p] * 3 + [None]),          # dq missing
        (z.make_shape(1, 1, 100, 64, 64, 3, 1, 64, "f32"), [p] * 6 + [None] + [p] * 4 + [None]),
        (z.make_shape(1, 1, 1024, 64, 64, 4, 1, 256, "f32"), [p] * 6 + [None] + [p] * 4 + [None]),
    ]
    for shape, ptrs in cases:
        rc_na = lib.zeco_gla_bwd_noalloc(ctypes.byref(shape), *ptrs, None)
        rc_ws = lib.zeco_gla_bwd(ctypes.byref(shape), *ptrs, ws, ctypes.c_size_t(64), None)
        assert rc_na == rc_ws and rc_na in (z.ZECO_ERR_ARG, z.ZECO_ERR_UNSUPPORTED), \
            (rc_na, rc_ws)
