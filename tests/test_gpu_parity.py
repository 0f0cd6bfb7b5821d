"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

fp32 I/O: max relative error (normwise infinity) <= 1e-4 per output tensor.
bf16 I/O: relative L2 error <= 2e-2 per output tensor.
Inputs come from the seeded generators in workloads.py; the oracle sees the
same (rounded) values widened to fp64.
"""
import numpy as np
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


def _assert(errs, dtype, what=""):
    t = parity.tol(dtype)
    bad = {k: v for k, v in errs.items() if not v <= t}
    assert not bad, f"{what} errors above {t}: {bad} (all: {errs})"


# ------------------------------------------------------------- tiny fp32


def test_tiny_f32_workload_full(z):
    """B1 H2 T1024 P4 C64 K2 d=64, fp32: every output, every state, fwd and bwd."""
    w = workloads.TINY_F32
    x = workloads.make_inputs(w)
    errs = parity.compare_full(z, x, w.P, w.K, w.C, "f32")
    _assert(errs, "f32", w.name)


@pytest.mark.parametrize("P,K,C", [(1, 1, 64), (2, 4, 32), (8, 2, 16), (32, 8, 16),
                                   (4, 32, 128), (16, 1, 32)])
def test_f32_invariance_to_P_K_C(z, P, K, C):
    """Every (P, K, C) grouping gives the recurrence's result (incl. P = T/C)."""
    x = workloads.make_custom(2, 1, 512, 32, 64, dtype="f32", seed=P * 100 + K * 10 + C,
                              s0_scale=0.5)
    errs = parity.compare_full(z, x, P, K, C, "f32")
    _assert(errs, "f32", f"P={P} K={K} C={C}")


def test_bf16_tensor_core_results_do_not_depend_on_K(z):
    """The segment scans run on K blocks of d_k rows (the pages' pipelined All-Scan
    granularity); every row's scan is the same arithmetic whatever the block, so
    the tensor-core path gives bit-identical outputs for every K."""
    B, H, T, dk, dv, P = 1, 2, 2048, 128, 256, 4
    x = workloads.make_custom(B, H, T, dk, dv, dtype="bf16", seed=41, qk_scale=1 / 16,
                              s0_scale=0.3)
    ref = None
    for K in (1, 2, 4, 8):
        assert z.resolve_path(z.make_shape(B, H, T, dk, dv, P, K, 64, "bf16", "tc")) == "tc"
        res = parity.run_gpu(z, x, P, K, 64, path="tc")
        res.pop("saved")
        if ref is None:
            ref = res
            continue
        for n, t in res.items():
            assert torch.equal(t, ref[n]), f"K={K}: {n} differs from K=1"


@pytest.mark.parametrize("case", ["no_decay", "slow_decay", "fast_decay", "single_chunk",
                                  "ragged_tiles", "min_width", "no_init_no_dsf"])
def test_f32_edge_cases(z, case):
    kw = dict(B=1, H=2, T=256, dk=64, dv=64, dtype="f32", seed=7, s0_scale=0.3)
    P, K, C = 4, 2, 32
    if case == "no_decay":
        kw["g_zero"] = True
    elif case == "slow_decay":
        kw["x_mean"] = 8.0
    elif case == "fast_decay":
        kw["x_mean"] = -6.0
        kw["x_scale"] = 2.0
    elif case == "single_chunk":
        kw.update(T=64)
        P, K, C = 1, 1, 64
    elif case == "ragged_tiles":
        kw.update(dk=48, dv=96, T=384)  # d_k tile of 64 and d_v slab of 64 both ragged
        P, K, C = 3, 3, 32
    elif case == "min_width":
        kw.update(dk=16, dv=32, T=128, B=3, H=1)
        P, K, C = 2, 1, 16
    x = workloads.make_custom(**kw)
    if case == "no_init_no_dsf":
        x["S0"] = None
        x["dS_final"] = None
    errs = parity.compare_full(z, x, P, K, C, "f32")
    _assert(errs, "f32", case)


def test_f32_full_width_and_long_segments(z):
    """d_k = 256, d_v = 512 (the GLA-1B head shape) in fp32, several 256-token segments."""
    x = workloads.make_custom(1, 1, 1024, 256, 512, dtype="f32", seed=21, qk_scale=1 / 16,
                              s0_scale=0.1)
    errs = parity.compare_full(z, x, 4, 8, 64, "f32", check_states=True)
    _assert(errs, "f32", "full width")


def test_repeated_calls_are_deterministic(z):
    w = workloads.TINY_F32
    x = workloads.make_inputs(w)
    a = parity.run_gpu(z, x, w.P, w.K, w.C)
    b = parity.run_gpu(z, x, w.P, w.K, w.C)
    for n in ("o", "S_final", "dq", "dk", "dv", "dlog_alpha", "dS0"):
        assert torch.equal(a[n], b[n]), n


# ------------------------------------------------------------------ bf16


@pytest.mark.parametrize("path", ["simt", "auto"])
def test_bf16_moderate_full(z, path):
    """bf16, GLA-1B head widths, several segments and chunks: every output."""
    x = workloads.make_custom(1, 2, 2048, 256, 512, dtype="bf16", seed=5, qk_scale=1 / 16,
                              s0_scale=0.1)
    errs = parity.compare_full(z, x, 4, 4, 64, "bf16", path=path)
    _assert(errs, "bf16", path)


@pytest.mark.parametrize("path", ["simt", "auto"])
def test_bf16_slow_decay_carry_dominated(z, path):
    """Slow decay: the state carried across segments dominates the outputs, so an
    error in the segment scan cannot hide under the intra-chunk terms."""
    x = workloads.make_custom(1, 2, 2048, 128, 256, dtype="bf16", seed=6, qk_scale=1 / 12,
                              x_mean=8.0, s0_scale=0.5)
    errs = parity.compare_full(z, x, 8, 2, 64, "bf16", path=path)
    _assert(errs, "bf16", path)
    # outputs of the first chunk of every segment only (the carry's share is largest there)
    res = parity.run_gpu(z, x, 8, 2, 64, path=path, bwd=False)
    ro, _ = oracle.gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"])
    L = 2048 // 8
    idx = np.concatenate([np.arange(p * L, p * L + 64) for p in range(8)])
    e = parity.rel_l2(parity.to_np(res["o"])[:, :, idx], ro[:, :, idx])
    assert e <= parity.TOL_BF16, e


@pytest.mark.parametrize("B,H,T,dk,dv,P,K", [(2, 1, 1024, 128, 128, 16, 2),
                                             (1, 2, 512, 256, 256, 8, 4),
                                             (1, 1, 4096, 128, 384, 2, 1),
                                             (1, 1, 256, 256, 512, 4, 8),
                                             (1, 2, 2048, 256, 128, 4, 2),
                                             (1, 1, 2048, 256, 384, 2, 4),
                                             (1, 2, 1024, 64, 64, 4, 2),
                                             (1, 1, 2048, 64, 512, 2, 1),
                                             (2, 1, 1024, 128, 192, 4, 2),
                                             (1, 1, 1024, 256, 320, 2, 4),
                                             (1, 1, 1024, 64, 448, 2, 2)])
def test_bf16_tensor_core_path_shapes(z, B, H, T, dk, dv, P, K):
    """The tcgen05 path on several tilings: one token block per segment (L = 64),
    d_v tiles of 128 and 256, one and several d_k tiles, several batches.  Every
    d_v (128, 256, 384, 512) runs dq, dk and dlog_alpha on the tensor-core kernel.
    d_k = 64 and d_v not a multiple of 128 (64, 192, 320, 448): partial tiles that
    read zeros past the end of the operands and store only what exists."""
    shape = z.make_shape(B, H, T, dk, dv, P, K, 64, "bf16", "tc")
    assert z.resolve_path(shape) == "tc"
    x = workloads.make_custom(B, H, T, dk, dv, dtype="bf16", seed=T + dk + dv,
                              qk_scale=1 / 16, s0_scale=0.2)
    names, _ = parity.kernel_names(z, lambda: parity.run_gpu(z, x, P, K, 64, path="tc"))
    assert "tc_bwd_dq" in names and "tc_bwd_dk" in names, names
    assert not any(n.startswith("simt") for n in names), names
    errs = parity.compare_full(z, x, P, K, 64, "bf16", path="tc")
    _assert(errs, "bf16", f"tc B{B} H{H} T{T} dk{dk} dv{dv} P{P}")


def _random_tc_shapes(n, seed=2026):
    """Seeded shapes on the tensor-core path's grid: d_k in {64, 128, 256}, d_v a
    multiple of 64, a few segments of a few chunks, K dividing d_k."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        dk = int(rng.choice([64, 128, 256]))
        dv = int(64 * rng.integers(1, 9))
        P = int(rng.choice([1, 2, 4]))
        L = int(64 * rng.integers(1, 5))
        K = int(rng.choice([k for k in (1, 2, 4, 8) if dk % k == 0]))
        out.append((int(rng.integers(1, 3)), int(rng.integers(1, 3)), P * L, dk, dv, P, K))
    return out


@pytest.mark.parametrize("B,H,T,dk,dv,P,K", _random_tc_shapes(10))
def test_bf16_tensor_core_random_shapes(z, B, H, T, dk, dv, P, K):
    """Seeded random shapes across the tensor-core grid (full and partial d_k and
    d_v tiles, 1-4 chunks per segment, several batches and heads) against the
    oracle, every output and state."""
    shape = z.make_shape(B, H, T, dk, dv, P, K, 64, "bf16", "tc")
    assert z.resolve_path(shape) == "tc"
    x = workloads.make_custom(B, H, T, dk, dv, dtype="bf16", seed=T + dk + dv + P,
                              qk_scale=1 / 16, s0_scale=0.2)
    names, _ = parity.kernel_names(z, lambda: parity.run_gpu(z, x, P, K, 64, path="tc"))
    assert not any(n.startswith("simt") for n in names), names
    errs = parity.compare_full(z, x, P, K, 64, "bf16", path="tc")
    _assert(errs, "bf16", f"tc random B{B} H{H} T{T} dk{dk} dv{dv} P{P} K{K}")


@pytest.mark.parametrize("dk,dv", [(256, 512), (64, 128)])
def test_bf16_chunk_128_runs_as_chunk_64_on_tensor_cores(z, dk, dv):
    """A bf16 call asking for C = 128 is evaluated with the tensor-core kernels'
    C = 64 (exact for any chunk length; a 128-token chunk's decay range implies
    that of its halves): every kernel is a tensor-core one and every output is
    bit-identical to the C = 64 call's, which the oracle checks."""
    B, H, T, P, K = 1, 2, 2048, 2, 4
    assert z.resolve_path(z.make_shape(B, H, T, dk, dv, P, K, 128, "bf16", "tc")) == "tc"
    x = workloads.make_custom(B, H, T, dk, dv, dtype="bf16", seed=dk + dv, qk_scale=1 / 16,
                              s0_scale=0.2)
    names, r128 = parity.kernel_names(z, lambda: parity.run_gpu(z, x, P, K, 128))
    assert "tc_bwd_dq" in names and not any(n.startswith("simt") for n in names), names
    r64 = parity.run_gpu(z, x, P, K, 64)
    for n in ("o", "S_final", "dq", "dk", "dv", "dlog_alpha", "dS0"):
        assert torch.equal(r128[n], r64[n]), n
    errs = parity.compare_full(z, x, P, K, 128, "bf16")
    _assert(errs, "bf16", f"C = 128 as 64, dk {dk} dv {dv}")


def test_f32_chunk_128_beyond_the_cuda_core_width_runs_as_chunk_64(z):
    """fp32 at d_k = 256 with C = 128: a 128-token chunk does not fit the CUDA-core
    kernels' shared memory at this width, so the call runs at C = 64 (forcing the
    SIMT path keeps C = 128 and is refused): identical to the C = 64 call and
    within the fp32 tolerance of the oracle."""
    B, H, T, dk, dv, P, K = 1, 1, 512, 256, 64, 2, 4
    with pytest.raises(z.ZecoError):
        z.resolve_path(z.make_shape(B, H, T, dk, dv, P, K, 128, "f32", "simt"))
    x = workloads.make_custom(B, H, T, dk, dv, dtype="f32", seed=6, s0_scale=0.3)
    r128 = parity.run_gpu(z, x, P, K, 128)
    r64 = parity.run_gpu(z, x, P, K, 64)
    for n in ("o", "S_final", "dq", "dk", "dv", "dlog_alpha", "dS0"):
        assert torch.equal(r128[n], r64[n]), n
    errs = parity.compare_full(z, x, P, K, 128, "f32")
    _assert(errs, "f32", "f32 C = 128 as 64, dk 256")


def test_bf16_chunk_128_off_the_tensor_core_grid_runs_as_chunk_64(z):
    """d_k = 192, d_v = 96 at C = 128: the CUDA-core steps run at C = 64 too (a
    128-token chunk would not fit their shared memory at this width): identical to
    the C = 64 call and to the oracle."""
    B, H, T, dk, dv, P, K = 1, 1, 1024, 192, 96, 2, 2
    x = workloads.make_custom(B, H, T, dk, dv, dtype="bf16", seed=5, qk_scale=1 / 16,
                              s0_scale=0.2)
    r128 = parity.run_gpu(z, x, P, K, 128)
    r64 = parity.run_gpu(z, x, P, K, 64)
    for n in ("o", "S_final", "dq", "dk", "dv", "dlog_alpha", "dS0"):
        assert torch.equal(r128[n], r64[n]), n
    errs = parity.compare_full(z, x, P, K, 128, "bf16")
    _assert(errs, "bf16", "C = 128 as 64, dk 192 dv 96")


@pytest.mark.parametrize("dk,dv,C", [(192, 512, 64), (64, 128, 32)])
def test_bf16_tensor_core_segment_states_with_cuda_core_sweeps(z, dk, dv, C):
    """Shapes whose segment states run on tensor cores (a partial d_k tile of 64
    rows: d_k = 192, or d_k = 64 with C = 32) while the sweeps run on CUDA cores."""
    shape = z.make_shape(1, 2, 2048, dk, dv, 2, 1, C, "bf16", "tc")
    assert z.resolve_path(shape) == "tc"
    x = workloads.make_custom(1, 2, 2048, dk, dv, dtype="bf16", seed=dk + dv + C,
                              qk_scale=1 / 16, s0_scale=0.2)
    names, _ = parity.kernel_names(z, lambda: parity.run_gpu(z, x, 2, 1, C, path="tc"))
    assert "tc_chunk_state" in names and "tc_dstate_local" in names, names
    errs = parity.compare_full(z, x, 2, 1, C, "bf16", path="tc")
    _assert(errs, "bf16", f"tc states, simt sweeps dk{dk} dv{dv} C{C}")


@pytest.mark.parametrize("B,H,T,dk,P,K", [(1, 1, 384, 256, 2, 8),    # 3 chunks per segment
                                         (1, 2, 640, 128, 2, 4),    # 5 chunks per segment
                                         (2, 1, 896, 256, 2, 2)])   # 7 chunks per segment
def test_bf16_odd_chunk_counts_in_the_dq_dk_sweeps(z, B, H, T, dk, P, K):
    """The dq/dk sweeps give alternate chunks to two epilogue groups and pass the
    dlog_alpha suffix between them: segments with an odd number of chunks leave
    the first group with the last chunk."""
    shape = z.make_shape(B, H, T, dk, 512, P, K, 64, "bf16", "tc")
    assert z.resolve_path(shape) == "tc"
    assert z.segments(shape) == P  # too short to be split further
    x = workloads.make_custom(B, H, T, dk, 512, dtype="bf16", seed=T + dk, qk_scale=1 / 16,
                              s0_scale=0.2)
    errs = parity.compare_full(z, x, P, K, 64, "bf16", path="tc")
    _assert(errs, "bf16", f"tc odd chunks B{B} H{H} T{T} dk{dk} P{P}")


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_overlap_schedules_give_identical_results(z, mode):
    # the default (mode 4: mode 1 plus the dq/dk sweeps on a high-priority
    # stream beside the dv sweep), the scan-independent passes on a second
    # stream (mode 1), the scan on a second stream (mode 2), pass 2 per block
    # of segments as soon as the scan reaches it (mode 3) or all on one stream
    # (mode 0): the same kernels on the same inputs, so bit-identical outputs
    w = workloads.LONG_FWDBWD.replace(T=16384, P=4)
    x = workloads.make_inputs(w)
    lib = z.load_library()
    a = parity.run_gpu(z, x, w.P, w.K, w.C)
    assert lib.zeco_set_overlap(mode) == z.ZECO_OK
    try:
        b = parity.run_gpu(z, x, w.P, w.K, w.C)
    finally:
        lib.zeco_set_overlap(z.OVERLAP_DEFAULT)
    for n in ("o", "S_final", "dq", "dk", "dv", "dlog_alpha", "dS0"):
        assert torch.equal(a[n], b[n]), n


def test_two_host_threads_with_their_own_streams(z):
    # the default schedule forks to auxiliary streams that belong to the calling host
    # thread: two threads running fwd+bwd at once, each on its own stream and inputs,
    # get exactly what one thread gets running them one after the other
    import threading
    ws = [workloads.LONG_FWDBWD.replace(T=8192, P=4, seed=s) for s in (11, 12)]
    xs = [{n: (t.cuda() if t is not None else None) for n, t in workloads.make_inputs(w).items()}
          for w in ws]
    w = ws[0]

    def run(x, stream):
        o, sf, saved = z.zeco_gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], P=w.P,
                                      K=w.K, C=w.C, stream=stream)
        g = z.zeco_gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], saved, x["do"],
                           x["dS_final"], P=w.P, K=w.K, C=w.C, stream=stream)
        return dict(o=o, S_final=sf, **{k: t for k, t in g.items() if t is not None})

    serial = []
    for x in xs:
        serial.append(run(x, torch.cuda.Stream()))
        torch.cuda.synchronize()
    results, errors = [None, None], []

    def worker(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(3):
                    results[i] = run(xs[i], st)
            st.synchronize()
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    z.check_device_status()
    for i in range(2):
        for n, t in serial[i].items():
            assert torch.equal(results[i][n], t), (i, n)


def test_forward_backward_replayed_from_a_cuda_graph(z):
    # the calls fork to their auxiliary streams and join back with events only, so a
    # forward+backward captured on one stream replays as a graph, bit for bit
    w = workloads.LONG_FWDBWD.replace(T=8192, P=4, seed=21)
    x = {n: (t.cuda() if t is not None else None) for n, t in workloads.make_inputs(w).items()}
    shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype)
    st = torch.cuda.Stream()
    o = torch.empty_like(x["v"])
    sf = torch.empty_like(x["S0"])
    saved = torch.empty(z.saved_bytes(shape), dtype=torch.uint8, device="cuda")
    ws = torch.empty(max(z.workspace_bytes(shape, True), 16), dtype=torch.uint8, device="cuda")
    grads = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]),
                 dv=torch.empty_like(x["v"]), dlog_alpha=torch.empty_like(x["log_alpha"]),
                 dS0=torch.empty_like(x["S0"]))

    def step():
        z.zeco_gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], P=w.P, K=w.K, C=w.C,
                       o=o, S_final=sf, saved=saved, stream=st)
        z.zeco_gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], saved, x["do"], x["dS_final"],
                       P=w.P, K=w.K, C=w.C, grads=grads, workspace=ws, stream=st)

    with torch.cuda.stream(st):
        step()  # eager (also creates the auxiliary streams before the capture)
    st.synchronize()
    ref = dict(o=o.clone(), S_final=sf.clone(), **{k: t.clone() for k, t in grads.items()})
    for t in (o, sf, *grads.values()):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    z.check_device_status()
    got = dict(o=o, S_final=sf, **grads)
    for n, t in ref.items():
        assert torch.equal(got[n], t), n


# ------------------------------------------------------------ decay forms


def _decay_case(z, decay, dtype, B, H, T, dk, dv, P, K, path):
    x = workloads.make_custom(B, H, T, dk, dv, dtype=dtype, seed=T + dk + 7 * decay,
                              qk_scale=1 / 16 if dtype == "bf16" else None, s0_scale=0.2)
    name = {oracle.DECAY_SCALAR: "scalar", oracle.DECAY_NONE: "none"}[decay]
    g = x["log_alpha"][..., 0].contiguous() if decay == oracle.DECAY_SCALAR else None
    dev = {n: (t.cuda() if t is not None else None) for n, t in x.items()}
    gd = g.cuda() if g is not None else None
    o, sf, saved = z.zeco_gla_fwd(dev["q"], dev["k"], dev["v"], gd, dev["S0"], P=P, K=K, C=64,
                                  path=path, decay=name)
    gr = z.zeco_gla_bwd(dev["q"], dev["k"], dev["v"], gd, saved, dev["do"], dev["dS_final"],
                        P=P, K=K, C=64, path=path, decay=name)
    torch.cuda.synchronize()
    np_in = {n: (parity.to_np(t) if t is not None else None) for n, t in x.items()}
    gn = parity.to_np(g) if g is not None else None
    ro, rsf = oracle.gla_fwd_decay(np_in["q"], np_in["k"], np_in["v"], gn, np_in["S0"], decay)
    rg = oracle.gla_bwd_decay(np_in["q"], np_in["k"], np_in["v"], gn, np_in["S0"], np_in["do"],
                              np_in["dS_final"], decay)
    errs = {"o": parity.err(parity.to_np(o), ro, dtype),
            "S_final": parity.err(parity.to_np(sf), rsf, dtype)}
    for n in ("dq", "dk", "dv", "dS0"):
        errs[n] = parity.err(parity.to_np(gr[n]), rg[n], dtype)
    if decay == oracle.DECAY_SCALAR:
        assert gr["dlog_alpha"].shape == (B, H, T)
        errs["dlog_alpha"] = parity.err(parity.to_np(gr["dlog_alpha"]), rg["dlog_alpha"], dtype)
    else:
        assert gr["dlog_alpha"] is None
    return errs


@pytest.mark.parametrize("decay", [1, 2])
def test_f32_decay_forms(z, decay):
    errs = _decay_case(z, decay, "f32", 1, 2, 1024, 64, 64, 4, 2, "auto")
    _assert(errs, "f32", f"f32 decay form {decay}")


@pytest.mark.parametrize("dk,dv", [(128, 512), (256, 512), (128, 256), (256, 128), (64, 64),
                                   (64, 192)])
@pytest.mark.parametrize("decay", [1, 2])
def test_bf16_decay_forms_on_tensor_cores(z, decay, dk, dv):
    # the tensor-core kernels read the scalar log-decay once per token (none for
    # the no-decay form): no [B,H,T,dk] broadcast is made, and the scalar
    # gradient is the sum of the reverse sweep's per-32-row partials (d_v < 512:
    # the dq/dk clusters' CTAs past d_v hold zero states)
    shape = z.make_shape(1, 2, 2048, dk, dv, 2, 4, 64, "bf16", "tc", decay)
    assert z.resolve_path(shape) == "tc"
    names, errs = parity.kernel_names(
        z, lambda: _decay_case(z, decay, "bf16", 1, 2, 2048, dk, dv, 2, 4, "tc"))
    _assert(errs, "bf16", f"bf16 tc decay form {decay} dk {dk} dv {dv}")
    assert "tc_decay" in names and "tc_bwd_dk" in names, names
    assert "expand_log_alpha" not in names and "reduce_dlog_alpha" not in names, names
    assert ("sum_dlog_alpha_parts" in names) == (decay == 1), names


def test_bf16_scalar_decay_broadcast_on_tensor_core_path(z):
    # C = 32: the tensor-core segment states, but the CUDA-core sweeps, which
    # take the log-decay broadcast to [B,H,T,dk]
    B, H, T, dk, dv, P, K, C = 1, 1, 1024, 128, 128, 2, 4, 32
    shape = z.make_shape(B, H, T, dk, dv, P, K, C, "bf16", "tc", 1)
    assert z.resolve_path(shape) == "tc"
    x = workloads.make_custom(B, H, T, dk, dv, dtype="bf16", seed=41, qk_scale=1 / 16,
                              s0_scale=0.2)
    g = x["log_alpha"][..., 0].contiguous()
    dev = {n: (t.cuda() if t is not None else None) for n, t in x.items()}

    def run():
        o, sf, saved = z.zeco_gla_fwd(dev["q"], dev["k"], dev["v"], g.cuda(), dev["S0"], P=P,
                                      K=K, C=C, path="tc", decay="scalar")
        gr = z.zeco_gla_bwd(dev["q"], dev["k"], dev["v"], g.cuda(), saved, dev["do"],
                            dev["dS_final"], P=P, K=K, C=C, path="tc", decay="scalar")
        torch.cuda.synchronize()
        return o, sf, gr

    names, (o, sf, gr) = parity.kernel_names(z, run)
    assert names.count("expand_log_alpha") == 2 and "reduce_dlog_alpha" in names, names
    assert "tc_decay" not in names, names
    np_in = {n: (parity.to_np(t) if t is not None else None) for n, t in x.items()}
    gn = parity.to_np(g)
    ro, rsf = oracle.gla_fwd_decay(np_in["q"], np_in["k"], np_in["v"], gn, np_in["S0"], 1)
    rg = oracle.gla_bwd_decay(np_in["q"], np_in["k"], np_in["v"], gn, np_in["S0"], np_in["do"],
                              np_in["dS_final"], 1)
    errs = {"o": parity.err(parity.to_np(o), ro, "bf16"),
            "S_final": parity.err(parity.to_np(sf), rsf, "bf16")}
    for n in ("dq", "dk", "dv", "dS0", "dlog_alpha"):
        errs[n] = parity.err(parity.to_np(gr[n]), rg[n], "bf16")
    _assert(errs, "bf16", "bf16 tc path, C = 32, scalar decay (broadcast)")


# ------------------------------------------------------------ segment counts


@pytest.mark.parametrize("dtype,dv,path", [("bf16", 512, "tc"), ("f32", 64, "simt")])
def test_one_chunk_per_segment(z, dtype, dv, path):
    # P = T / C: every segment is one chunk, the scans carry 128 steps
    B, H, T, dk = 1, 1, 8192, 128 if dtype == "bf16" else 64
    P, K = T // 64, 4
    x = workloads.make_custom(B, H, T, dk, dv, dtype=dtype, seed=5,
                              qk_scale=1 / 16 if dtype == "bf16" else None, s0_scale=0.2)
    shape = z.make_shape(B, H, T, dk, dv, P, K, 64, dtype, path)
    assert z.segments(shape) == P
    errs = parity.compare_full(z, x, P, K, 64, dtype, path=path)
    _assert(errs, dtype, f"P = T/C ({path})")


def test_low_parallelism_shape_is_split_and_unchanged(z):
    # one segment of 16K tokens, 2 heads: 2 x 4 d_v tiles per segment, so the
    # library evaluates 32 sub-segments of 512 tokens (256 CTAs); the outputs
    # match the oracle as for any split
    B, H, T, dk, dv = 1, 2, 16384, 128, 512
    shape = z.make_shape(B, H, T, dk, dv, 1, 1, 64, "bf16", "auto")
    assert z.segments(shape) == 32
    x = workloads.make_custom(B, H, T, dk, dv, dtype="bf16", seed=6, qk_scale=1 / 16,
                              s0_scale=0.2)
    errs = parity.compare_full(z, x, 1, 1, 64, "bf16")
    _assert(errs, "bf16", "P = 1 split")


# ------------------------------------- edge cases on the tensor-core dq/dk kernel


def _tc_edge_inputs(case, dk=128, dv=512, device="cpu"):
    kw = dict(B=1, H=2, T=2048, dk=dk, dv=dv, dtype="bf16", seed=31, qk_scale=1 / 12,
              s0_scale=0.3, device=device)
    if case == "slow_decay":
        kw.update(x_mean=8.0, s0_scale=0.5)   # log_alpha ~ -2e-5: the carry dominates
    elif case == "fast_decay":
        kw.update(x_mean=-18.0)               # log_alpha ~ -1.1: chunk sums near -72
    elif case == "no_decay":
        kw.update(g_zero=True)                # log_alpha = 0 exactly
    return workloads.make_custom(**kw)


@pytest.mark.parametrize("dk,dv", [(128, 512), (64, 64)])
@pytest.mark.parametrize("case", ["slow_decay", "fast_decay", "no_decay"])
def test_bf16_tc_dq_dk_kernel_edge_cases(z, case, dk, dv):
    """The decay regimes the method has, on the tensor-core dq/dk/dlog_alpha
    kernel (d_v = 512, and d_k = d_v = 64 with its partial tiles): the
    carry-dominated slow decay, a fast decay whose chunk log-decay sums reach
    about -72 (the chunk factorisation's range ends at -80), and exactly no
    decay.  Besides every full tensor, the first and last two chunks of every
    segment are checked on their own: there the states carried across segments
    (forward) and back (adjoint) weigh most."""
    B, H, T, P, K = 1, 2, 2048, 8, 2
    shape = z.make_shape(B, H, T, dk, dv, P, K, 64, "bf16", "tc")
    assert z.resolve_path(shape) == "tc"
    x = _tc_edge_inputs(case, dk, dv)
    csum = x["log_alpha"].float().view(B, H, T // 64, 64, dk).sum(3)
    if case == "fast_decay":
        assert -80.0 < float(csum.min()) and float(csum.max()) < -60.0
    names, res = parity.kernel_names(z, lambda: parity.run_gpu(z, x, P, K, 64, path="tc"))
    assert "tc_bwd_dq" in names and "tc_bwd_dk" in names, names
    ro, rsf = oracle.gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"])
    rg = oracle.gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], x["do"],
                        x["dS_final"])
    errs = {"o": parity.rel_l2(parity.to_np(res["o"]), ro),
            "S_final": parity.rel_l2(parity.to_np(res["S_final"]), rsf)}
    for n in ("dq", "dk", "dv", "dlog_alpha", "dS0"):
        errs[n] = parity.rel_l2(parity.to_np(res[n]), rg[n])
    idx = parity.chunk_rows(T, z.segments(shape))
    for n, r in (("o", ro), ("dq", rg["dq"]), ("dk", rg["dk"]), ("dv", rg["dv"]),
                 ("dlog_alpha", rg["dlog_alpha"])):
        errs[n + "[segment ends]"] = parity.rel_l2(parity.to_np(res[n])[:, :, idx],
                                                   r[:, :, idx])
    _assert(errs, "bf16", f"tc {case} dk {dk} dv {dv}")


@pytest.mark.parametrize("x_mean", [0.0, 8.0])
def test_bf16_tc_whole_16k_token_segments(z, x_mean):
    """Segments of L = 16,384 tokens on the tensor-core path, as in the 1M-token
    workload (38 sequences of one segment each fill one wave, so the library
    does not split them): the dlog_alpha suffix sums run over all 16K tokens of a
    segment.  The first and last sequences are checked in full."""
    B, H, T, dk, dv = 38, 1, 16384, 128, 512
    shape = z.make_shape(B, H, T, dk, dv, 1, 1, 64, "bf16", "tc")
    assert z.resolve_path(shape) == "tc"
    assert z.segments(shape) == 1
    x = workloads.make_custom(B, H, T, dk, dv, dtype="bf16", seed=16, qk_scale=1 / 16,
                              x_mean=x_mean, s0_scale=0.3, device="cuda")
    names, res = parity.kernel_names(z, lambda: parity.run_gpu(z, x, 1, 1, 64, path="tc"))
    assert "tc_bwd_dq" in names and "tc_bwd_dk" in names, names
    errs = {}
    for b in (0, B - 1):
        xs = {n: t[b:b + 1].cpu() for n, t in x.items()}
        ro, rsf = oracle.gla_fwd(xs["q"], xs["k"], xs["v"], xs["log_alpha"], xs["S0"])
        rg = oracle.gla_bwd(xs["q"], xs["k"], xs["v"], xs["log_alpha"], xs["S0"], xs["do"],
                            xs["dS_final"])
        errs[f"o[{b}]"] = parity.rel_l2(parity.to_np(res["o"][b:b + 1]), ro)
        errs[f"S_final[{b}]"] = parity.rel_l2(parity.to_np(res["S_final"][b:b + 1]), rsf)
        for n in ("dq", "dk", "dv", "dlog_alpha", "dS0"):
            errs[f"{n}[{b}]"] = parity.rel_l2(parity.to_np(res[n][b:b + 1]), rg[n])
    _assert(errs, "bf16", f"L=16384 x_mean={x_mean}")
