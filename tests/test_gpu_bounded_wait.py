"""The bounded device waits of the tensor-core kernels, exercised on the GPU
without a fault: a diagnostic kernel of four warps waits 64 times per thread on
mbarriers that nothing will complete.  The first wait must give up within its
time limit and the others at once after it (the CTA's abort word), so the
kernel ends after about one time limit; the timeout must be reported by the
status calls, and the context must stay usable."""
import time

import pytest
import torch

import oracle
import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def z():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_state_scan_gb300 import build
    build.build()
    import chunked_state_scan_gb300 as pkg
    pkg.load_library()
    return pkg


def test_wait_that_cannot_complete_gives_up_and_is_reported(z):
    lib = z.load_library()
    torch.cuda.synchronize()
    assert lib.zeco_check_device_status() == z.ZECO_OK  # nothing pending
    t0 = time.perf_counter()
    z.selftest_bounded_wait()
    torch.cuda.synchronize()  # returns: the kernel gave up instead of hanging
    dt = time.perf_counter() - t0
    # 4 warps x 64 waits that never complete cost about one 2 s limit in all
    assert 1.5 <= dt <= 10.0, dt
    assert lib.zeco_check_device_status() == z.ZECO_ERR_TIMEOUT
    assert lib.zeco_check_device_status() == z.ZECO_OK  # read and cleared
    # the context is still usable: a small forward matches the oracle
    w = workloads.TINY_F32
    x = workloads.make_inputs(w)
    g = {n: t.cuda() for n, t in x.items()}
    o, sf, _ = z.zeco_gla_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["S0"], P=w.P, K=w.K,
                              C=w.C)
    torch.cuda.synchronize()
    ro, rsf = oracle.gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"])
    assert parity.err(parity.to_np(o), ro, "f32") <= parity.tol("f32")
    assert parity.err(parity.to_np(sf), rsf, "f32") <= parity.tol("f32")


def test_last_device_status_synchronises_its_stream(z):
    # zeco_last_device_status(stream) waits for the stream's work itself: the
    # diagnostic is launched on a side stream and the status is read with no
    # synchronisation by the caller
    torch.cuda.synchronize()
    assert z.last_device_status() == z.ZECO_OK
    side = torch.cuda.Stream()
    t0 = time.perf_counter()
    z.selftest_bounded_wait(side)
    rc = z.last_device_status(side)
    dt = time.perf_counter() - t0
    assert rc == z.ZECO_ERR_TIMEOUT, rc
    assert 1.5 <= dt <= 10.0, dt
    assert z.last_device_status(side) == z.ZECO_OK  # read and cleared
