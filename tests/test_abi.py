"""The C-ABI library: builds, loads, exports what the header declares, and
rejects bad arguments on the host (no GPU work is launched here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from chunked_state_scan_gb300 import build
    build.build()
    import chunked_state_scan_gb300 as z
    return z.load_library()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(zeco_\w+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "zeco_gla_fwd" in names and "zeco_gla_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


def _shape(**kw):
    import chunked_state_scan_gb300 as z
    a = dict(B=1, H=4, T=1 << 20, dk=256, dv=512, P=64, K=8, C=64, dtype="bf16")
    a.update(kw)
    return z.make_shape(**a)


def test_sizes_follow_the_layout(lib):
    import chunked_state_scan_gb300 as z
    s = _shape()
    state = 4 * 65 * 256 * 512 * 4
    gam = 4 * 64 * 256 * 4
    # tensor-core path: the forward keeps Q~ and K~ (bf16), e^{b_last} per 64-token
    # chunk (fp32) and the masked intra-chunk scores [B,H,T,64] (bf16) in `saved`
    decay = (2 * 4 * (1 << 20) * 256 * 2 + 4 * (1 << 20) // 64 * 256 * 4
             + 4 * (1 << 20) * 64 * 2)
    assert z.saved_bytes(s) == state + gam + decay
    assert z.saved_bytes(_shape(path="simt")) == state + gam
    qdq = 4 * (1 << 20) * 256 * 4
    # backward only: the masked intra-chunk score gradients [B,H,T,64] bf16
    dA = 4 * (1 << 20) * 64 * 2
    assert z.workspace_bytes(s, True) == state + gam + qdq + dA
    assert z.workspace_bytes(s, False) == 0
    # decay forms on the tensor-core path: read in their own layout, so no
    # broadcast scratch; the scalar backward adds its fp32 gradient partials
    # [dk / 32][B,H,T]
    parts = (256 // 32) * 4 * (1 << 20) * 4
    assert z.workspace_bytes(_shape(decay="scalar"), False) == 0
    assert z.workspace_bytes(_shape(decay="none"), False) == 0
    assert z.workspace_bytes(_shape(decay="scalar"), True) == state + gam + qdq + dA + parts
    assert z.workspace_bytes(_shape(decay="none"), True) == state + gam + qdq + dA
    # elsewhere the log-decay is broadcast to [B,H,T,dk] (and its per-row
    # gradient too, in the backward)
    bc = 4 * (1 << 20) * 256 * 2
    assert z.workspace_bytes(_shape(decay="scalar", path="simt"), False) == bc
    # (C = 32: the tensor-core segment states, the CUDA-core sweeps)
    assert z.workspace_bytes(_shape(decay="scalar", C=32, dk=128, dv=128, K=4), False) == bc // 2
    # the SIMT path keeps no decay-weighted operands
    simt = _shape(path="simt", dtype="f32", dk=64, dv=64)
    st64 = 4 * 65 * 64 * 64 * 4
    assert z.workspace_bytes(simt, False) == 0
    # (+ the CUDA-core dq/dk kernel's intra-chunk dA [B,H,T,C] fp32)
    assert z.workspace_bytes(simt, True) == (st64 + 4 * 64 * 64 * 4 + 4 * (1 << 20) * 64 * 4
                                             + 4 * (1 << 20) * 64 * 4)


@pytest.mark.parametrize("kw,code", [
    (dict(T=1000), -1),            # T not divisible by P
    (dict(P=3), -1),
    (dict(K=3), -1),               # dk % K != 0
    (dict(C=48), -1),              # L % C != 0
    (dict(C=8, T=8 * 64), -2),     # C outside {16,32,64,128}
    (dict(dk=272), -2),
    (dict(dv=48), -2),
    (dict(dv=1024), -2),
    (dict(B=0), -1),
    (dict(dtype=7), -1),
])
def test_invalid_shapes_are_rejected(lib, kw, code):
    s = _shape(**kw)
    if kw.get("dtype") == 7:
        s.dtype = 7
    assert lib.zeco_gla_saved_bytes(ctypes.byref(s)) == 0
    assert lib.zeco_gla_resolve_path(ctypes.byref(s)) == code
    rc = lib.zeco_gla_fwd(ctypes.byref(s), *([ctypes.c_void_p(256)] * 4), None,
                          ctypes.c_void_p(256), None, ctypes.c_void_p(256), None, 0, None)
    assert rc == code


def test_null_and_misaligned_pointers_are_rejected(lib):
    s = _shape(T=4096, P=4)
    ok = ctypes.c_void_p(4096)
    bad = ctypes.c_void_p(4100)
    args = [ok] * 4
    assert lib.zeco_gla_fwd(ctypes.byref(s), *args, None, None, None, ok, None, 0, None) == -1
    assert lib.zeco_gla_fwd(ctypes.byref(s), bad, ok, ok, ok, None, ok, None, ok, None, 0,
                            None) == -1
    # forward with the scalar decay form off the tensor-core sweeps (it needs
    # scratch for the broadcast log-decay): workspace missing, then too small
    sc = _shape(T=4096, P=4, decay="scalar", path="simt")
    assert lib.zeco_gla_fwd(ctypes.byref(sc), *args, None, ok, None, ok, None, 0, None) == -1
    assert lib.zeco_gla_fwd(ctypes.byref(sc), *args, None, ok, None, ok, ok, 16, None) == -3
    # workspace too small for the backward
    rc = lib.zeco_gla_bwd(ctypes.byref(s), ok, ok, ok, ok, ok, ok, None, ok, ok, ok, ok, None,
                          ok, 16, None)
    assert rc == -3
    assert lib.zeco_strerror(-3) == b"workspace too small"
    assert lib.zeco_strerror(12345) == b"unknown error code"


def test_path_resolution(lib):
    import chunked_state_scan_gb300 as z
    assert z.resolve_path(_shape(dtype="f32", dk=64, dv=64, T=1024, P=4, K=2)) == "simt"
    # fp32 at full width does not fit the SIMT kernels' shared memory with C=128
    with pytest.raises(z.ZecoError):
        z.resolve_path(_shape(dtype="f32", C=128, path="simt"))
    # nor does bf16 on the CUDA-core path; on the tensor-core path a bf16 call with
    # C = 128 is evaluated at the kernels' C = 64 (results do not depend on C), with
    # the same scratch sizes and segment count
    with pytest.raises(z.ZecoError):
        z.resolve_path(_shape(C=128, path="simt"))
    for path in ("tc", "auto"):
        s128, s64 = _shape(C=128, path=path), _shape(C=64, path=path)
        assert z.resolve_path(s128) == "tc"
        assert z.saved_bytes(s128) == z.saved_bytes(s64)
        assert z.workspace_bytes(s128, True) == z.workspace_bytes(s64, True)
        assert z.segments(s128) == z.segments(s64)
    assert z.resolve_path(_shape(C=128, dk=128, dv=128, K=4)) == "tc"
    # shorter chunks are kept as asked (their decay range may be what the caller
    # needs): C = 32 takes the tensor-core segment states and the CUDA-core sweeps
    # (GPU tests check which kernels run)
    assert z.resolve_path(_shape(C=32, dk=128, dv=128, K=4)) == "tc"


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 512), (128, 192), (256, 320), (64, 448),
                                   (192, 512), (256, 512)])
def test_bf16_shapes_resolve_to_the_tensor_core_path(lib, dk, dv):
    """Every bf16 shape with C = 64 and d_k, d_v multiples of 64 runs on the
    tensor-core path (d_k = 192 with its sweeps on CUDA cores); others on the
    CUDA-core path."""
    import chunked_state_scan_gb300 as z
    assert z.resolve_path(_shape(T=4096, P=4, K=1, dk=dk, dv=dv)) == "tc"
    assert z.resolve_path(_shape(T=4096, P=4, K=1, dk=dk, dv=dv, path="simt")) == "simt"


@pytest.mark.parametrize("dk,dv", [(96, 128), (128, 96), (32, 32)])
def test_bf16_shapes_off_the_64_grid_take_the_cuda_core_path(lib, dk, dv):
    import chunked_state_scan_gb300 as z
    assert z.resolve_path(_shape(T=4096, P=4, K=1, dk=dk, dv=dv)) == "simt"
    with pytest.raises(z.ZecoError):
        z.resolve_path(_shape(T=4096, P=4, K=1, dk=dk, dv=dv, path="tc"))


def test_decay_forms_workspace_and_arguments(lib):
    import chunked_state_scan_gb300 as z
    diag = _shape(T=4096, P=4, path="simt")
    for name in ("scalar", "none"):
        s = _shape(T=4096, P=4, decay=name, path="simt")
        extra = 4 * 4096 * 256 * 2  # broadcast log-decay [B,H,T,dk] bf16
        assert z.workspace_bytes(s, False) == z.workspace_bytes(diag, False) + extra
        assert z.workspace_bytes(s, True) == z.workspace_bytes(diag, True) + 2 * extra
    ok = ctypes.c_void_p(4096)
    # without decay log_alpha may be NULL (the call then fails only on the tiny
    # workspace); with decay it may not
    none = _shape(T=4096, P=4, decay="none", path="simt")
    assert lib.zeco_gla_fwd(ctypes.byref(none), ok, ok, ok, None, None, ok, None, ok, ok, 16,
                            None) == -3
    assert lib.zeco_gla_fwd(ctypes.byref(diag), ok, ok, ok, None, None, ok, None, ok, ok, 16,
                            None) == -1
    bad = _shape(T=4096, P=4)
    bad.decay = 3
    assert lib.zeco_gla_resolve_path(ctypes.byref(bad)) == -1


def test_grid_limits(lib):
    import chunked_state_scan_gb300 as z
    # (b, h, segment) goes on grid x: B*H*P beyond 65,535 is supported ...
    assert z.segments(_shape(T=1 << 20, P=16384, K=8)) == 16384          # 65,536 segments
    assert z.segments(_shape(B=8, H=32, T=65536, P=256, K=8)) == 256      # 65,536
    # ... up to (2^31 - 1) / 32; the scans put B*H on grid z (65,535 at most)
    for kw in (dict(B=2048, H=16, T=2048 * 64, P=2048, K=8),             # B*H*P = 2^26
               dict(B=256, H=256, T=64, P=1, K=8)):                     # B*H = 65,536
        with pytest.raises(z.ZecoError):
            z.segments(_shape(**kw))


def test_segment_count_fills_the_gpu(lib):
    import chunked_state_scan_gb300 as z
    # the 1M-token workload already gives 1024 CTAs: no split
    assert z.segments(_shape()) == 64
    # GLA-1B layer shape with one segment: 16 sub-segments of 1024 tokens
    assert z.segments(_shape(T=16384, P=1, K=1)) == 16
    # 8-segment forward at 131K tokens: split in two
    assert z.segments(_shape(T=131072, P=8, K=4)) == 16
    # the saved buffer follows the effective count
    s = _shape(T=16384, P=1, K=1, path="simt")
    assert z.saved_bytes(s) == 4 * 17 * 256 * 512 * 4 + 4 * 16 * 256 * 4
    # too short to split (fewer than 4 chunks per sub-segment)
    assert z.segments(_shape(T=512, P=2, K=8)) == 2


def test_noalloc_shape_errors_match_the_workspace_backward(lib):
    # invalid and unsupported shapes return zeco_gla_bwd's codes before any CUDA call
    import chunked_state_scan_gb300 as z
    cases = [z.make_shape(1, 1, 100, 64, 64, 3, 1, 64, "f32"),      # T % P != 0
             z.make_shape(1, 1, 1024, 64, 64, 4, 1, 256, "f32"),    # C outside the set
             z.make_shape(1, 1, 1024, 64, 1024, 4, 1, 64, "f32"),   # d_v too wide
             z.make_shape(0, 1, 1024, 64, 64, 4, 1, 64, "f32")]     # B = 0
    for shape in cases:
        rc_na = lib.zeco_gla_bwd_noalloc(ctypes.byref(shape), *([None] * 13))
        rc_ws = lib.zeco_gla_bwd(ctypes.byref(shape), *([None] * 12), None, 0, None)
        assert rc_na == rc_ws < 0, (rc_na, rc_ws)


def test_binding_rejects_bad_tensors_before_the_library():
    """The binding hands raw pointers to the library, so it checks every tensor
    first: device, contiguity, dtype, shape and buffer size."""
    import torch
    import chunked_state_scan_gb300 as z
    q = torch.zeros(1, 2, 128, 64)
    with pytest.raises(ValueError, match="CUDA"):
        z.zeco_gla_fwd(q, q, q, q, P=1, K=1, C=64)
    with pytest.raises(ValueError, match="CUDA"):
        z.zeco_gla_bwd(q, q, q, q, torch.zeros(16, dtype=torch.uint8), q, P=1, K=1, C=64)
    cpu = torch.device("cpu")
    z._expect(q, "q", cpu, q.shape, torch.float32)  # a matching tensor passes
    z._expect(None, "S0", cpu)                       # optional tensors may be absent
    with pytest.raises(ValueError, match="required"):
        z._expect(None, "k", cpu, optional=False)
    with pytest.raises(ValueError, match="contiguous"):
        z._expect(q.transpose(2, 3), "k", cpu)
    with pytest.raises(ValueError, match="dtype"):
        z._expect(q.half(), "k", cpu, q.shape, torch.float32)
    with pytest.raises(ValueError, match="shape"):
        z._expect(q[:, :1].contiguous(), "k", cpu, q.shape, torch.float32)
    with pytest.raises(ValueError, match="bytes"):
        z._expect(torch.zeros(10, dtype=torch.uint8), "saved", cpu, nbytes=11)
    with pytest.raises(ValueError, match="expected cuda"):
        z._expect(q, "k", torch.device("cuda", 0))
    with pytest.raises(TypeError):
        z._expect([1, 2], "k", cpu)


def test_schedule_and_profiling_switches_on_the_host(lib):
    """zeco_set_overlap takes the modes 0-4 only; the profiling switch records
    nothing while it is off (no GPU work: no call is enqueued)."""
    import chunked_state_scan_gb300 as z
    try:
        for bad in (-1, 5, 1 << 20):
            assert lib.zeco_set_overlap(bad) == z.ZECO_ERR_ARG
        for mode in range(5):
            assert lib.zeco_set_overlap(mode) == z.ZECO_OK
    finally:
        assert lib.zeco_set_overlap(z.OVERLAP_DEFAULT) == z.ZECO_OK
    lib.zeco_set_profile_events.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.zeco_profile_kernel_name.restype = ctypes.c_char_p
    assert lib.zeco_set_profile_events(None, 0) == z.ZECO_OK
    assert lib.zeco_profile_event_count() == 0
    assert lib.zeco_profile_kernel_name(0) is None
    assert lib.zeco_profile_kernel_name(-1) is None


def test_every_accepted_shape_runs_under_auto(lib):
    """With path AUTO every width and chunk length the boundary accepts resolves
    to a path (C = 128 runs at C = 64 where that is what runs it); forcing the
    CUDA-core path keeps C = 128, which its shared memory holds up to d_k = 128."""
    import chunked_state_scan_gb300 as z
    refused_auto, refused_simt = [], []
    for dtype in ("bf16", "f32"):
        for dk in range(16, 257, 16):
            for dv in range(32, 513, 32):
                for C in (16, 32, 64, 128):
                    for path, out in (("auto", refused_auto), ("simt", refused_simt)):
                        try:
                            z.resolve_path(_shape(dtype=dtype, T=16384, P=4, K=1, dk=dk, dv=dv,
                                                  C=C, path=path))
                        except z.ZecoError:
                            out.append((dtype, dk, C))
    assert not refused_auto, refused_auto[:5]
    assert sorted(set(refused_simt)) == sorted(
        (dt, dk, 128) for dt in ("bf16", "f32") for dk in range(144, 257, 16))
