"""GPU parity at the full workload sizes, on sampled outputs.

The throughput workloads are too large for a full fp64 oracle run, so the
oracle computes selected output columns (o, dv and the state columns) and
selected d_k rows (dq, dk, dlog_alpha, dS0) exactly, one by one: every column
and every row of the state follows its own recurrence.  The GPU side runs the
whole workload in the same launch configuration that bench.py times.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import parity

pytestmark = pytest.mark.gpu

COLS = [0, 131, 258, 511]
ROWS = [3, 200]


@pytest.fixture(scope="module")
def z():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_state_scan_gb300 import build
    build.build()
    import chunked_state_scan_gb300 as pkg
    pkg.load_library()
    return pkg


def _sample_check(z, w, heads, with_bwd, COLS=COLS, ROWS=ROWS):
    dev = "cuda"
    x = workloads.make_inputs(w, device=dev)
    o, sf, saved = z.zeco_gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], P=w.P,
                                  K=w.K, C=w.C)
    grads = None
    if with_bwd:
        grads = z.zeco_gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], saved, x["do"],
                               x["dS_final"], P=w.P, K=w.K, C=w.C)
    torch.cuda.synchronize()
    pe = z.segments(z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype))
    states = parity.saved_states(saved, w.B, w.H, pe, w.dk, w.dv)
    errs = {}
    for b, h in heads:
        sl = lambda t: t[b:b + 1, h:h + 1].cpu()  # noqa: E731
        xs = {n: sl(t) for n, t in x.items()}
        ro, rsf = oracle.gla_fwd(xs["q"], xs["k"], xs["v"], xs["log_alpha"], xs["S0"],
                                 cols=COLS)
        errs[f"o[{b},{h}]"] = parity.rel_l2(parity.to_np(o[b, h][:, COLS]), ro[0, 0])
        errs[f"S_final[{b},{h}]"] = parity.rel_l2(parity.to_np(sf[b, h][:, COLS]), rsf[0, 0])
        bs = oracle.boundary_states_cols(xs["q"], xs["k"], xs["v"], xs["log_alpha"], xs["S0"],
                                         pe, COLS)
        errs[f"S_in[{b},{h}]"] = parity.rel_l2(parity.to_np(states[b, h][..., COLS]), bs[0, 0])
        if with_bwd:
            rg = oracle.gla_bwd(xs["q"], xs["k"], xs["v"], xs["log_alpha"], xs["S0"], xs["do"],
                                xs["dS_final"], rows=ROWS, cols=COLS)
            for n in ("dq", "dk", "dlog_alpha"):
                errs[f"{n}[{b},{h}]"] = parity.rel_l2(parity.to_np(grads[n][b, h][:, ROWS]),
                                                      rg[n][0, 0])
            errs[f"dv[{b},{h}]"] = parity.rel_l2(parity.to_np(grads["dv"][b, h][:, COLS]),
                                                 rg["dv"][0, 0])
            errs[f"dS0[{b},{h}]"] = parity.rel_l2(parity.to_np(grads["dS0"][b, h][ROWS]),
                                                  rg["dS0"][0, 0])
    bad = {k: v for k, v in errs.items() if not v <= parity.TOL_BF16}
    assert not bad, f"{w.name}: {bad} (all: {errs})"
    del x, o, sf, saved, grads
    torch.cuda.empty_cache()


def test_gla1b_fwd_sampled(z):
    _sample_check(z, workloads.GLA1B_FWD, [(0, 0), (0, 3)], with_bwd=True)


def test_segmented_fwd_sampled(z):
    _sample_check(z, workloads.SEG_FWD, [(0, 1)], with_bwd=False)


def test_batched_fwdbwd_sampled(z):
    _sample_check(z, workloads.BATCHED_FWDBWD, [(0, 0), (7, 3)], with_bwd=True)


def test_long_fwdbwd_sampled(z):
    _sample_check(z, workloads.LONG_FWDBWD, [(0, 2)], with_bwd=True)


def test_more_than_65535_segment_blocks_sampled(z):
    # B*H*P = 65,536 (P = T/C: one chunk per segment): the (b, h, segment) index
    # of every kernel lives on grid x, so the shape runs like any other
    w = workloads.LONG_FWDBWD.replace(name="grid_x_H8_T524288_P8192", H=8, T=1 << 19, dk=128,
                                      dv=128, P=8192, K=4)
    assert z.segments(z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype)) == 8192
    _sample_check(z, w, [(0, 0), (0, 7)], with_bwd=True, COLS=[0, 77, 127], ROWS=[3, 100])


def test_small_head_fwdbwd_sampled(z):
    # d_k = 64, d_v = 128 at the 1M-token size: partial 128-row tiles in the
    # segment-state and dq/dk kernels, native d_k = 64 sweeps
    w = workloads.SMALL_HEAD_FWDBWD
    assert z.resolve_path(z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C,
                                       w.dtype)) == "tc"
    _sample_check(z, w, [(0, 1)], with_bwd=True, COLS=[0, 63, 64, 127], ROWS=[0, 31, 63])
