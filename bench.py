"""Throughput of segmented GLA forward+backward on one GB300 (per rank).

Workload (default): the 1M-token, 64-segment forward+backward --
B=1, H=4, T=1,048,576, P=64 (L=16,384), C=64, K=8, d_k=256, d_v=512, bf16 I/O,
fp32 accumulation, synthetic inputs from workloads.py.  One step is one
zeco_gla_fwd plus one zeco_gla_bwd over the whole batch (every kernel of the
path).  Inputs (14 GiB) are far larger than the 126 MB L2, so no L2 flush is
needed between steps (workloads whose inputs are under ~0.5 GB get an untimed
L2 flush before every timed step).

Timing: W untimed warm-up steps, then K timed steps bracketed by a barrier and
torch.cuda.synchronize() on both sides, CUDA events on the library's stream,
maximum over ranks.  N > 1 (torchrun) runs N independent replicas, one per GPU
(weak scaling; the library has no cross-GPU exchange).

Other modes: `--secondary` prints one line per secondary workload (GLA-1B layer
forward, 8-segment forward, batched forward+backward); `--scan-sweep` times the
segment scans at many segments; `--schedule-sweep` times the schedules of the work
beside the scan at many segments; `--forms` times the step in each decay form;
`--impl reference` times the fp64 CPU oracle instead, on a bounded sample of the same
workload, on this host's cores.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "GLA fwd+bwd tokens/sec on 1 GB300 and % of roofline (1M tok, P=64)"

# HBM bytes per token per head (bf16, d_k=256, d_v=512), per kernel, in two
# accountings.  Segment states are counted per token as state_bytes / L.
#   method: the bytes of the method's own tensors that the step a kernel carries
#     out must move -- its inputs (q, k, v, log_alpha, do, segment states) read
#     once and its outputs (o, dq, dk, dv, dlog_alpha, segment states) written
#     once; intermediates this implementation keeps (Q~, K~, e^{b_last}, A, dA,
#     q.dq) count zero.  The roofline fraction of a kernel is taken on these.
#   impl: what the kernel actually reads and writes, intermediates included.
# The ZeCO operator total (fwd 5632 + bwd 8192 B per token-head, plus segment
# states) is the roofline denominator of the whole step.
E = 2  # bytes per bf16 element


def _state(dk, dv, L):
    return dk * dv * 4 / L  # one fp32 dk x dv state per segment, per token


def kernel_bytes_per_token(dk, dv, L, e=E, C=64):
    """Implementation bytes per token-head of every kernel (what it moves)."""
    st = _state(dk, dv, L)
    eb = dk * 4 / C       # e^{b_last}: one fp32 row per chunk, per token
    return {
        # pass 1: read K~, v, e^{b_last}; write one local state per segment
        "chunk_state": e * (dk + dv) + eb + st,
        "seg_scan_fwd": 2 * st,
        # decay pass: read q, k, g; write Q~, K~ and e^{b_last}
        "decay": e * 5 * dk + eb,
        # intra-chunk scores: read Q~, K~; write the masked A (64 per token)
        "A": e * (2 * dk + C),
        # pass 2: read Q~, K~, A, v, e^{b_last} and S_in[p]; write o
        "fwd_out": e * (2 * dk + 2 * dv + C) + eb + st,
        # bwd pre-pass: read Q~, do, e^{b_last}; write one adjoint state per segment
        "dstate_local": e * (dk + dv) + eb + st,
        "seg_scan_rev": 3 * st,
        # dv: read Q~, K~, A, do, e^{b_last} and D[p+1]; write dv
        "bwd_dv": e * (2 * dk + 2 * dv + C) + eb + st,
        # dq, dk, dg (one launch, CUDA-core path): read q, k, v, g, do, S_in[p], D[p+1];
        # write dq, dk, dg
        "bwd_dqk": e * (3 * dk + 2 * dv) + e * 3 * dk + 2 * st,
        # intra-chunk score gradients: read do, v; write the masked dA (64 per token)
        "dA": e * (2 * dv + C),
        # dq sweep: read Q~, K~, g, v, do, dA, e^{b_last} and S_in[p]; write dq, q.dq (fp32)
        "bwd_dq": e * (3 * dk + 2 * dv + C) + eb + e * dk + 4 * dk + st,
        # dk sweep: read Q~, K~, g, v, do, dA, e^{b_last}, q.dq, D[p+1]; write dk, dlog_alpha
        "bwd_dk": e * (3 * dk + 2 * dv + C) + eb + 4 * dk + 2 * e * dk + st,
    }


def method_bytes_per_token(dk, dv, L, e=E):
    """The method's bytes per token-head for the step each kernel carries out."""
    st = _state(dk, dv, L)
    return {
        "chunk_state": e * (2 * dk + dv) + st,        # k, g, v -> S_loc
        "seg_scan_fwd": 2 * st,                       # S_loc, S_in
        "decay": e * 3 * dk,                          # q, k, g (outputs are intermediates)
        "A": 0.0,                                     # intermediates only
        "fwd_out": e * (3 * dk + 2 * dv) + st,        # q, k, g, v, S_in -> o
        "dstate_local": e * (2 * dk + dv) + st,       # q, g, do -> dS_loc
        "seg_scan_rev": 3 * st,
        "bwd_dv": e * (3 * dk + 2 * dv) + st,         # q, k, g, do, D -> dv
        "bwd_dqk": e * (3 * dk + 2 * dv) + e * 3 * dk + 2 * st,
        "dA": e * 2 * dv,                             # v, do (output is an intermediate)
        "bwd_dq": e * (3 * dk + 2 * dv) + e * dk + st,       # q, k, g, v, do, S_in -> dq
        "bwd_dk": e * (3 * dk + 2 * dv) + 2 * e * dk + st,   # q, k, g, v, do, D -> dk, dg
    }


def zeco_operator_bytes_per_token(dk, dv, L, e=E, bwd=True):
    """ZeCO two-pass algorithmic bytes per token-head (fwd [+ bwd] + segment states)."""
    fwd = e * (5 * dk + 3 * dv)
    if not bwd:
        return fwd + 16 * dk * dv / L
    bwd_b = e * (8 * dk + 4 * dv)
    states = (16 + 20) * dk * dv / L
    return fwd + bwd_b + states


def zeco_operator_flops_per_token(dk, dv, C, bwd=True):
    fwd = 2 * C * (dk + dv) + 6 * dk * dv
    if not bwd:
        return fwd
    return fwd + 2 * C * (3 * dk + 2 * dv) + 12 * dk * dv


def canonical_kernel(name):
    if name == "tc_A":
        return "A"
    for key in ("chunk_state", "seg_scan_fwd", "decay", "fwd_out", "dstate_local",
                "seg_scan_rev", "bwd_dv", "dA", "bwd_dqk", "bwd_dq", "bwd_dk"):
        if key in name:
            return key
    return name


def measured_traffic(path, kernel, impl_bytes):
    """DRAM bytes of one launch of `kernel` from the committed ncu capture
    (profiles/traffic.json): the launch's implementation bytes `impl_bytes` times
    the captured ratio of DRAM traffic to implementation bytes; None when there is
    no capture or the kernel's sources changed since it was taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            ent = json.load(f).get(f"{path}:{kernel}")
    except (OSError, ValueError):
        return None
    if not ent or not ent.get("impl_bytes_per_token_head"):
        return None
    for rel, digest in ent.get("sources", {}).items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return impl_bytes * ent["bytes_per_token_head"] / ent["impl_bytes_per_token_head"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


# ------------------------------------------------------------ clocks sampler


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------- distributed


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(elapsed_s_max: float, tokens_per_rank_step: int, steps: int, world: int):
    """Whole-job throughput: tokens processed by all ranks / the slowest rank's time."""
    total = tokens_per_rank_step * steps * world
    return total / elapsed_s_max, elapsed_s_max * 1e3 / steps


# ------------------------------------------------------------- CPU oracle leg


def cpu_oracle_sample(w, sample_tokens, nthreads=None):
    """Time the fp64 oracle (fwd, + full bwd when the workload has a backward) on
    the first `sample_tokens` tokens of every head of batch 0.  Returns tokens/s in
    the workload's unit and details."""
    import oracle
    x = workloads.make_inputs(w.replace(T=sample_tokens, P=1, B=1), device="cpu")
    nt = nthreads or oracle.default_threads()
    t0 = time.perf_counter()
    oracle.gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], nthreads=nt)
    if w.bwd:
        oracle.gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], x["do"],
                       x["dS_final"], nthreads=nt)
    dt = time.perf_counter() - t0
    # all H heads of the sample were processed: the sample covers sample_tokens tokens
    return sample_tokens / dt, dt, nt


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle as it stands, on this host's cores.
    Each step is a bounded sample of the workload (the first ``--ref-sample-tokens``
    tokens of batch 0, all heads, forward + backward), so ``value`` is the oracle's
    rate on that sample and ``ms_per_step`` the measured time of one sample step."""
    if rank != 0:
        return 0
    import oracle
    w = workloads.BY_NAME[args.workload]
    sample = args.ref_sample_tokens
    for _ in range(args.warmup):  # loads the oracle library and warms its threads
        xs = workloads.make_inputs(w.replace(T=64, P=1, B=1), device="cpu")
        oracle.gla_fwd(xs["q"], xs["k"], xs["v"], xs["log_alpha"], xs["S0"])
    vals, times, nt = [], [], None
    for _ in range(args.steps):
        v, dt, nt = cpu_oracle_sample(w, sample)
        vals.append(v)
        times.append(dt)
    value = sum(vals) / len(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                   "P": w.P, "K": w.K, "C": w.C, "step_tokens": sample,
                   "step": f"a sample of the workload: batch 0, all {w.H} heads, the first "
                           f"{sample} tokens (the rate is tokens/s on that sample)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                         "sample": f"batch 0, all {w.H} heads, first {sample} tokens, fp64 "
                                   f"recurrence fwd + brute-force adjoint bwd, per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ GPU measurement


def profile_step(lib, step, dev, n_ev=64):
    """One step with the library's per-kernel start/end events.  Returns a list
    of (kernel, start_ms, end_ms) on one timeline (relative to the first start)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    for e in evs:
        e.record()  # materialise the handles
    torch.cuda.synchronize(dev)
    handles = (ctypes.c_void_p * n_ev)(*[e.cuda_event for e in evs])
    lib.zeco_set_profile_events.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.zeco_profile_kernel_name.restype = ctypes.c_char_p
    lib.zeco_set_profile_events(ctypes.cast(handles, ctypes.c_void_p), n_ev)
    try:
        step()
        n = lib.zeco_profile_event_count() // 2
        names = [lib.zeco_profile_kernel_name(i).decode() for i in range(n)]
    finally:
        lib.zeco_set_profile_events(None, 0)
    torch.cuda.synchronize(dev)
    base = evs[0]
    return [(names[i], base.elapsed_time(evs[2 * i]), base.elapsed_time(evs[2 * i + 1]))
            for i in range(n)]


def scan_overlap(intervals):
    """The pages' overlap instrument (Pith review, 'What would settle it'; Eq. 11):
    the share of the segment scan's time during which no diagonal-attention kernel
    (the intra-chunk scores A, forward; their gradient dA, backward) runs."""
    def span(name):
        return [(a, b) for n, a, b in intervals if canonical_kernel(n) == name]
    out = {}
    for direction, scan, diag in (("fwd", "seg_scan_fwd", "A"), ("bwd", "seg_scan_rev", "dA")):
        sc, dg = span(scan), span(diag)
        if not sc or not dg:
            continue
        s_len = sum(b - a for a, b in sc)
        ov = sum(max(0.0, min(b, d1) - max(a, d0)) for a, b in sc for d0, d1 in dg)
        out[direction] = {"scan_ms": s_len, "overlapped_ms": ov,
                          "non_overlapped_frac": 1.0 - ov / s_len if s_len > 0 else None}
    return out


def copy_bound(dev, nbytes=1 << 31):
    """Pinned host <-> device copy rates on this machine (GB/s): each direction alone
    and both at once (best of 3), the bound of any step that moves its inputs in
    and its outputs out."""
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s_up, s_dn = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(up, down):
        best = None
        for _ in range(3):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            if up:
                with torch.cuda.stream(s_up):
                    d_in.copy_(h_in, non_blocking=True)
            if down:
                with torch.cuda.stream(s_dn):
                    h_out.copy_(d_out, non_blocking=True)
            torch.cuda.synchronize(dev)
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        return nbytes / best / 1e9

    res = {"h2d_gbs": timed(True, False), "d2h_gbs": timed(False, True)}
    both = timed(True, True)  # each direction moved nbytes in that time
    res["both_each_gbs"] = both
    res["bytes"] = nbytes
    del h_in, h_out, d_in, d_out
    return res


def measure(w, args, world, rank, local, want_e2e=True, want_cpu=True, quiet=False):
    """Time ``args.steps`` steps of workload ``w`` (forward, plus the backward when the
    workload has one) and return the JSON line as a dict."""
    import chunked_state_scan_gb300 as z
    lib = z.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    x = workloads.make_inputs(w, device=dev)
    shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype, args.path)
    path = z.resolve_path(shape)
    # outputs and buffers, allocated once (the library itself never allocates)
    o = torch.empty_like(x["v"])
    S_final = torch.empty_like(x["S0"])
    saved = torch.empty(z.saved_bytes(shape), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(z.workspace_bytes(shape, True), 16), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(max(z.workspace_bytes(shape, False), 16), dtype=torch.uint8, device=dev)
    grads = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]),
                 dv=torch.empty_like(x["v"]), dlog_alpha=torch.empty_like(x["log_alpha"]),
                 dS0=torch.empty_like(x["S0"]))
    in_bytes = sum(t.numel() * t.element_size() for t in x.values())
    # inputs smaller than a few L2s (126 MB) could be served from L2 on the next
    # step: then L2 is flushed (a 512 MB write, untimed) before every timed step
    flush = in_bytes < 4 * 126e6
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if flush else None

    def step(xx=x):
        z.zeco_gla_fwd(xx["q"], xx["k"], xx["v"], xx["log_alpha"], xx["S0"], P=w.P, K=w.K,
                       C=w.C, path=args.path, o=o, S_final=S_final, saved=saved,
                       workspace=ws_f, stream=stream)
        if w.bwd:
            z.zeco_gla_bwd(xx["q"], xx["k"], xx["v"], xx["log_alpha"], saved, xx["do"],
                           xx["dS_final"], P=w.P, K=w.K, C=w.C, path=args.path, grads=grads,
                           workspace=ws, stream=stream)

    per_step = []  # device ms of each step of the last timed_steps call

    def timed_steps(n):
        """Device time of n steps (ms), L2 flushed before each when the inputs are small;
        each step's own time is left in per_step."""
        per_step.clear()
        if not flush:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
            evs[0].record(stream)
            for i in range(n):
                step()
                evs[i + 1].record(stream)
            torch.cuda.synchronize(dev)
            per_step.extend(evs[i].elapsed_time(evs[i + 1]) for i in range(n))
            return evs[0].elapsed_time(evs[n])
        for _ in range(n):
            with torch.cuda.stream(stream):
                flush_buf.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            per_step.append(e0.elapsed_time(e1))
        return sum(per_step)

    torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- per-kernel durations: start/end events of every kernel, with every
    #      kernel on one stream (zeco_set_overlap(0)), so that no kernel's time is
    #      stretched by another running beside it
    lib.zeco_set_overlap.argtypes = [ctypes.c_int]
    lib.zeco_set_overlap(0)
    try:
        prof = [profile_step(lib, step, dev) for _ in range(2)]
    finally:
        lib.zeco_set_overlap(z.OVERLAP_DEFAULT)
    per_kernel = {}
    for run in prof:
        for n, a, b in run:
            per_kernel.setdefault(n, []).append(b - a)
    kern_ms = {k: sum(v) / len(v) for k, v in per_kernel.items()}
    launches_per_step = len(prof[0])

    # ---- timed region
    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    elapsed = timed_steps(args.steps) / 1e3
    steps_ms = list(per_step)
    barrier(world)
    clk = clocks.stop()
    dev_status = lib.zeco_last_device_status(ctypes.c_void_p(stream.cuda_stream))
    elapsed_max = max_over_ranks(elapsed, world)
    value, ms_step = aggregate(elapsed_max, w.tokens, args.steps, world)

    # ---- the other schedules of the work beside the scan (zeco_set_overlap):
    #      0 = one stream, 1 = the score passes on a second stream, 2 = the scan on
    #      a second stream beside the diagonal attention (the pages' schedule), 3 =
    #      pass 2 per block of segments; the default (4) is the timed region above.
    #      The Eq. 11 instrument for each
    overlap = None
    if path == "tc":
        modes = {}
        try:
            for mode in (0, 1, 2, 3, z.OVERLAP_DEFAULT):
                lib.zeco_set_overlap(mode)
                step()
                torch.cuda.synchronize(dev)
                modes[mode] = (timed_steps(args.steps) / args.steps, profile_step(lib, step, dev))
        finally:
            lib.zeco_set_overlap(z.OVERLAP_DEFAULT)
        names = {0: "mode0_one_stream", 1: "mode1_aux_scores", 2: "mode2_aux_scan",
                 3: "mode3_pass2_per_segment_block", 4: "mode4_default_dqk_beside_dv"}
        step_ms = {names[m]: modes[m][0] for m in (0, 1, 2, 3)}
        step_ms[names[4]] = ms_step
        overlap = {
            "step_ms": step_ms,
            "scan_not_overlapped": {names[m]: scan_overlap(modes[m][1]) for m in (1, 2, 3, 4)},
            "note": "mode 4 (default, the timed region): mode 1, and in the backward the dq/dk "
                    "sweeps on a high-priority stream beside the dv sweep; mode 1: scores A / "
                    "dA on a second stream beside pass 1, the scans (and the dv sweep); mode "
                    "2: the segment scans on a second stream beside the A / dA pass; mode 3: "
                    "the forward scan in blocks of segments, pass 2 of each block on the "
                    "second stream as soon as its block is scanned; non_overlapped_frac = "
                    "share of the scan's kernel time with no A / dA kernel running (Eq. 11 "
                    "instrument)"}

    # ---- roofline of the dominant kernel and of the whole step
    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    bh = w.B * w.H
    kb = kernel_bytes_per_token(w.dk, w.dv, w.L)
    mb = method_bytes_per_token(w.dk, w.dv, w.L)
    dom = max(kern_ms, key=kern_ms.get)
    dom_key = canonical_kernel(dom)
    dom_bytes = mb.get(dom_key, 0.0) * w.T * bh
    dom_impl_bytes = kb.get(dom_key, 0.0) * w.T * bh
    dom_gbs = dom_bytes / (kern_ms[dom] * 1e-3) / 1e9
    op_bytes = zeco_operator_bytes_per_token(w.dk, w.dv, w.L, bwd=w.bwd) * w.T * bh
    op_flops = zeco_operator_flops_per_token(w.dk, w.dv, w.C, bwd=w.bwd) * w.T * bh
    t_roof = max(op_bytes / (hbm_peak * 1e9), op_flops / (float(peaks["bf16_tflops"]) * 1e12))
    step_s = ms_step * 1e-3
    traffic = measured_traffic(path, dom, dom_impl_bytes)
    # every kernel's bytes over its event-timed duration (GB/s), both accountings
    kern_gbs = {k: {"method": mb[canonical_kernel(k)] * w.T * bh / (ms * 1e-3) / 1e9,
                    "impl": kb[canonical_kernel(k)] * w.T * bh / (ms * 1e-3) / 1e9}
                for k, ms in kern_ms.items() if canonical_kernel(k) in kb and ms > 0}
    impl_total = sum(kb[canonical_kernel(k)] for k in kern_ms if canonical_kernel(k) in kb)
    method_total = zeco_operator_bytes_per_token(w.dk, w.dv, w.L, bwd=w.bwd)
    scan_ms = sum(v for k, v in kern_ms.items() if "seg_scan" in k)

    line = {
        "metric": METRIC if w.name == workloads.LONG_FWDBWD.name else
        f"GLA {'fwd+bwd' if w.bwd else 'fwd'} tokens/sec on 1 GB300 and % of roofline "
        f"({w.name})",
        "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "step_ms_stats": {"mean": statistics.fmean(steps_ms),
                          "std": statistics.stdev(steps_ms) if len(steps_ms) > 1 else 0.0,
                          "min": min(steps_ms), "max": max(steps_ms), "n": len(steps_ms),
                          "rank": rank},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; shapes and distributions of the GLA-1B layer workload)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                   "P": w.P, "K": w.K, "C": w.C, "path": path, "step": "fwd+bwd" if w.bwd
                   else "fwd", "segments_evaluated": z.segments(shape),
                   "l2": ("flushed before every timed step (512 MB write, untimed): inputs "
                          f"{in_bytes / 1e6:.0f} MB") if flush else
                   f"no flush: inputs {in_bytes / 2**30:.1f} GiB >> 126 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": dom_gbs, "peak": hbm_peak,
                     "unit": "GB/s", "frac": dom_gbs / hbm_peak, "traffic": traffic,
                     "traffic_unit": "DRAM bytes per launch (ncu capture of the small case: its "
                                     "traffic / implementation-bytes ratio times this launch's "
                                     "implementation bytes)",
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "algorithmic_bytes": "the method's inputs and outputs of this step "
                                          "(no intermediates)",
                     "impl_bytes_per_launch": dom_impl_bytes,
                     "impl_frac": dom_impl_bytes / (kern_ms[dom] * 1e-3) / 1e9 / hbm_peak},
        "operator_roofline": {"bytes": op_bytes, "flops": op_flops, "t_roof_ms": t_roof * 1e3,
                              "frac": t_roof / step_s,
                              "impl_bytes_per_token_head": impl_total,
                              "method_bytes_per_token_head": method_total,
                              "impl_over_method": impl_total / method_total,
                              "note": "ZeCO two-pass algorithmic bytes/flops per step vs "
                                      f"{peak_kind} peaks"},
        "device_status": "ok" if dev_status == 0 else f"error {dev_status}",
        "kernels_ms": kern_ms, "kernels_gbs": kern_gbs, "overlap": overlap,
        "scan_share": scan_ms / sum(kern_ms.values()),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }

    # ---- end to end through the public API with host buffers.  Every step uploads
    # its inputs from pinned host memory and downloads all its outputs; the steps
    # are pipelined the way a caller would run them: uploads and downloads have
    # their own streams, inputs and outputs are double-buffered on the device, so
    # step i+1's upload and step i-1's download overlap step i's kernels.  Each
    # tensor's copy may be cut into kCopyStreams contiguous pieces on as many
    # streams per direction (--e2e-copy-streams; default one: the host link, not
    # the copy engines, bounds the copies, and 1, 2, 4 or 8 streams measured
    # within 3% of each other, one the fastest).
    if want_e2e and w.bwd:
        names_in = ["q", "k", "v", "log_alpha", "do", "dS_final", "S0"]
        host_in = {n: x[n].cpu().pin_memory() for n in names_in}
        out_names = ("o", "S_final", "dq", "dk", "dv", "dlog_alpha", "dS0")
        out0 = dict(o=o, S_final=S_final, **grads)
        out1 = {n: torch.empty_like(t) for n, t in out0.items()}
        dev_out = [out0, out1]
        host_out = {n: torch.empty(out0[n].shape, dtype=out0[n].dtype, pin_memory=True)
                    for n in out_names}
        dev_in = [{n: torch.empty_like(x[n]) for n in names_in} for _ in range(2)]
        del x
        bi = sum(t.numel() * t.element_size() for t in host_in.values())
        bo = sum(t.numel() * t.element_size() for t in host_out.values())
        kCopyStreams = args.e2e_copy_streams
        s_up = [torch.cuda.Stream(device=dev) for _ in range(kCopyStreams)]
        s_down = [torch.cuda.Stream(device=dev) for _ in range(kCopyStreams)]
        ev_up = [[torch.cuda.Event() for _ in range(kCopyStreams)] for _ in range(2)]
        ev_run = [torch.cuda.Event() for _ in range(2)]
        ev_down = [[torch.cuda.Event() for _ in range(kCopyStreams)] for _ in range(2)]

        def pieces(t):  # kCopyStreams contiguous views of a contiguous tensor
            flat = t.view(-1)
            n = flat.numel()
            stp = -(-n // kCopyStreams)
            return [flat[c * stp:min(n, (c + 1) * stp)] for c in range(kCopyStreams)]

        def run_into(xx, od):
            z.zeco_gla_fwd(xx["q"], xx["k"], xx["v"], xx["log_alpha"], xx["S0"], P=w.P, K=w.K,
                           C=w.C, path=args.path, o=od["o"], S_final=od["S_final"], saved=saved,
                           workspace=ws_f, stream=stream)
            z.zeco_gla_bwd(xx["q"], xx["k"], xx["v"], xx["log_alpha"], saved, xx["do"],
                           xx["dS_final"], P=w.P, K=w.K, C=w.C, path=args.path,
                           grads={n: od[n] for n in ("dq", "dk", "dv", "dlog_alpha", "dS0")},
                           workspace=ws, stream=stream)

        up_pieces = [{nm: (pieces(dev_in[b][nm]), pieces(host_in[nm])) for nm in names_in}
                     for b in range(2)]
        down_pieces = [{nm: (pieces(host_out[nm]), pieces(dev_out[b][nm])) for nm in out_names}
                       for b in range(2)]

        def e2e_steps(n_steps):
            for i in range(n_steps):
                b = i % 2
                for c, su in enumerate(s_up):
                    with torch.cuda.stream(su):
                        if i >= 2:
                            su.wait_event(ev_run[b])  # step i-2 is done with these inputs
                        for nm in names_in:
                            dst, src = up_pieces[b][nm]
                            dst[c].copy_(src[c], non_blocking=True)
                        ev_up[b][c].record(su)
                for c in range(kCopyStreams):
                    stream.wait_event(ev_up[b][c])
                    if i >= 2:
                        stream.wait_event(ev_down[b][c])  # step i-2's outputs are downloaded
                run_into(dev_in[b], dev_out[b])
                ev_run[b].record(stream)
                for c, sd in enumerate(s_down):
                    with torch.cuda.stream(sd):
                        sd.wait_event(ev_run[b])
                        for nm in out_names:
                            dst, src = down_pieces[b][nm]
                            dst[c].copy_(src[c], non_blocking=True)
                        ev_down[b][c].record(sd)

        e2e_steps(2)
        torch.cuda.synchronize(dev)
        barrier(world)
        t0 = time.perf_counter()
        e2e_steps(args.e2e_steps)
        torch.cuda.synchronize(dev)
        t1 = time.perf_counter()
        barrier(world)
        el = max_over_ranks(t1 - t0, world)
        ev, _ = aggregate(el, w.tokens, args.e2e_steps, world)
        # the copy bound: a step cannot beat moving its bytes at this machine's pinned
        # copy rates (both directions at once), nor its own device time
        del dev_in, dev_out, out1, up_pieces, down_pieces
        torch.cuda.empty_cache()
        cb = copy_bound(dev)
        t_copy = max(bi / (cb["both_each_gbs"] * 1e9), bo / (cb["both_each_gbs"] * 1e9))
        bound = w.tokens * world / max(t_copy, step_s)
        line["e2e"] = {"value": ev, "unit": "tokens/s", "h2d_bytes_per_step": bi,
                       "d2h_bytes_per_step": bo, "steps": args.e2e_steps,
                       "copy_bound": {**cb, "t_copy_ms": t_copy * 1e3, "bound_tokens_s": bound,
                                      "frac": ev / bound},
                       "note": "uploads, kernels and downloads of consecutive steps pipelined "
                               f"(each tensor's copy in {kCopyStreams} pieces on "
                               f"{kCopyStreams} streams per direction); "
                               "every step's copies inside the timed region; copy_bound: plain "
                               "pinned copies of 2 GiB on this box"}

    # ---- CPU baseline (rank 0 only, N = 1 only)
    if want_cpu and rank == 0 and world == 1:
        sample = min(args.cpu_sample_tokens, w.T)
        v, dt, nt = cpu_oracle_sample(w, sample)
        line["cpu_baseline"] = {
            "value": v, "unit": "tokens/s", "cores": nt, "kind": "oracle",
            "sample": f"batch 0, all {w.H} heads, first {sample} tokens: fp64 "
                      f"token recurrence fwd" + (" + brute-force adjoint bwd" if w.bwd else "")
                      + f" ({dt:.1f} s)"}
    return line


def scan_sweep(args, local):
    """The segment scans at many segments (``--scan-sweep``): the 1M-token workload's
    inputs with P in {64, 1024, 4096, 8192, T/C}; each scan's time and bytes/s."""
    import chunked_state_scan_gb300 as z
    lib = z.load_library()
    dev = torch.device("cuda", local)
    peaks, peak_kind = load_peaks()
    base = workloads.LONG_FWDBWD
    x = workloads.make_inputs(base, device=dev)
    out = []
    for P in (64, 1024, 4096, 8192, base.T // base.C):
        w = base.replace(P=P, name=f"scan_sweep_P{P}")
        stream = torch.cuda.Stream(device=dev)
        shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype)
        saved = torch.empty(z.saved_bytes(shape), dtype=torch.uint8, device=dev)
        ws = torch.empty(z.workspace_bytes(shape, True), dtype=torch.uint8, device=dev)

        def step():
            _, _, _ = z.zeco_gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], P=P,
                                     K=w.K, C=w.C, saved=saved, stream=stream)
            z.zeco_gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], saved, x["do"],
                           x["dS_final"], P=P, K=w.K, C=w.C, workspace=ws, stream=stream)

        step()
        torch.cuda.synchronize(dev)
        lib.zeco_set_overlap.argtypes = [ctypes.c_int]
        lib.zeco_set_overlap(0)  # every kernel alone: the scans' own times
        try:
            runs = [profile_step(lib, step, dev) for _ in range(3)]
        finally:
            lib.zeco_set_overlap(z.OVERLAP_DEFAULT)
        kb = kernel_bytes_per_token(w.dk, w.dv, w.L)
        res = {"P": P, "L": w.L}
        for name in ("seg_scan_fwd", "seg_scan_rev"):
            ms = [b - a for r in runs for n, a, b in r if n == name]
            t = sum(ms) / len(ms)
            gbs = kb[name] * w.T * w.B * w.H / (t * 1e-3) / 1e9
            res[name] = {"ms": t, "gbs": gbs, "frac_of_hbm": gbs / float(peaks["hbm_gbs"])}
        out.append(res)
        del saved, ws
        torch.cuda.empty_cache()
    return {"scan_sweep": out, "peak_source": f"{peak_kind} hbm_gbs",
            "workload": base.name + " inputs, P varied"}


def schedule_sweep(args, local):
    """The headline workload's inputs cut into P segments, P from 64 to T/C
    (``--schedule-sweep``): the step time in schedules 0 (one stream), 1 (score passes
    on a second stream) and 4 (mode 1 plus dq/dk beside dv; the default runs it from 4
    chunks per segment up, one stream below), each set through zeco_set_overlap."""
    import chunked_state_scan_gb300 as z
    lib = z.load_library()
    dev = torch.device("cuda", local)
    base = workloads.LONG_FWDBWD
    x = workloads.make_inputs(base, device=dev)
    out = []
    lib.zeco_set_overlap.argtypes = [ctypes.c_int]
    for P in (64, 256, 1024, 4096, 8192, base.T // base.C):
        w = base.replace(P=P)
        shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype)
        saved = torch.empty(z.saved_bytes(shape), dtype=torch.uint8, device=dev)
        ws = torch.empty(z.workspace_bytes(shape, True), dtype=torch.uint8, device=dev)
        stream = torch.cuda.Stream(device=dev)

        def step():
            z.zeco_gla_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["S0"], P=P, K=w.K,
                           C=w.C, saved=saved, stream=stream)
            z.zeco_gla_bwd(x["q"], x["k"], x["v"], x["log_alpha"], saved, x["do"],
                           x["dS_final"], P=P, K=w.K, C=w.C, workspace=ws, stream=stream)

        res = {"P": P, "chunks_per_segment": w.L // w.C}
        try:
            for mode in (0, 1, 4):
                lib.zeco_set_overlap(mode)
                for _ in range(max(2, args.warmup)):
                    step()
                torch.cuda.synchronize(dev)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(args.steps):
                    step()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                key = "mode4_default_ms" if mode == 4 else f"mode{mode}_ms"
                res[key] = e0.elapsed_time(e1) / args.steps
        finally:
            lib.zeco_set_overlap(z.OVERLAP_DEFAULT)
        out.append(res)
        del saved, ws
        torch.cuda.empty_cache()
    return {"schedule_sweep": out, "workload": base.name + " inputs, P varied",
            "steps": args.steps}


def decay_forms(args, local):
    """The headline workload's fwd+bwd step in each decay form (``--forms``): per-token
    scalar and no decay beside the diagonal form, each with its step time (L2 flushed
    before every step when the inputs are small; here they are not) and the per-kernel
    times with every kernel on one stream."""
    import chunked_state_scan_gb300 as z
    lib = z.load_library()
    dev = torch.device("cuda", local)
    w = workloads.LONG_FWDBWD
    x = workloads.make_inputs(w, device=dev)
    stream = torch.cuda.Stream(device=dev)
    out = []
    for form in ("diag", "scalar", "none"):
        g = {"diag": x["log_alpha"], "scalar": x["log_alpha"][..., 0].contiguous(),
             "none": None}[form]
        shape = z.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.P, w.K, w.C, w.dtype, "auto", form)
        saved = torch.empty(z.saved_bytes(shape), dtype=torch.uint8, device=dev)
        ws = torch.empty(max(z.workspace_bytes(shape, True), 16), dtype=torch.uint8,
                         device=dev)
        ws_f = torch.empty(max(z.workspace_bytes(shape, False), 16), dtype=torch.uint8,
                           device=dev)
        o = torch.empty_like(x["v"])
        S_final = torch.empty_like(x["S0"])
        grads = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]),
                     dv=torch.empty_like(x["v"]),
                     dlog_alpha=torch.empty_like(g) if g is not None else None,
                     dS0=torch.empty_like(x["S0"]))

        def step():
            z.zeco_gla_fwd(x["q"], x["k"], x["v"], g, x["S0"], P=w.P, K=w.K, C=w.C, o=o,
                           S_final=S_final, saved=saved, workspace=ws_f, stream=stream,
                           decay=form)
            z.zeco_gla_bwd(x["q"], x["k"], x["v"], g, saved, x["do"], x["dS_final"], P=w.P,
                           K=w.K, C=w.C, grads=grads, workspace=ws, stream=stream, decay=form)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        lib.zeco_set_overlap.argtypes = [ctypes.c_int]
        lib.zeco_set_overlap(0)
        try:
            runs = [profile_step(lib, step, dev) for _ in range(3)]
        finally:
            lib.zeco_set_overlap(z.OVERLAP_DEFAULT)
        kms = {}
        for r in runs:
            for n, a, b in r:
                kms[n] = kms.get(n, 0.0) + (b - a) / len(runs)
        out.append({"decay": form, "ms_per_step": ms, "tokens_per_s": w.tokens / (ms * 1e-3),
                    "workspace_bytes_bwd": z.workspace_bytes(shape, True),
                    "kernels_ms": kms})
        del saved, ws, ws_f, grads, o, S_final
        torch.cuda.empty_cache()
    return {"decay_forms": out, "workload": w.name, "steps": args.steps, "warmup": args.warmup}


# ---------------------------------------------------------------- main


SECONDARY = [workloads.GLA1B_FWD.name, workloads.SEG_FWD.name, workloads.BATCHED_FWDBWD.name]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=workloads.LONG_FWDBWD.name)
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="streams (and pieces of each tensor's copy) per direction in e2e")
    ap.add_argument("--cpu-sample-tokens", type=int, default=16384)
    ap.add_argument("--ref-sample-tokens", type=int, default=4096)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--secondary", action="store_true",
                    help="one JSON line per secondary workload (GLA-1B layer fwd, "
                         "8-segment fwd, batched fwd+bwd) instead of the headline")
    ap.add_argument("--scan-sweep", action="store_true",
                    help="time the segment scans at P in {64, 1024, 4096, 8192, T/C}")
    ap.add_argument("--schedule-sweep", action="store_true",
                    help="time schedules 0, 1 and 4 at P from 64 to T/C")
    ap.add_argument("--forms", action="store_true",
                    help="time the headline step in the diagonal, scalar and no-decay forms")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl != "reference":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import chunked_state_scan_gb300 as z
    z.load_library()
    if args.scan_sweep or args.forms or args.schedule_sweep:
        res = (scan_sweep(args, local) if args.scan_sweep else
               decay_forms(args, local) if args.forms else schedule_sweep(args, local))
        if rank == 0:
            print(json.dumps(res), flush=True)
        return 0
    names = SECONDARY if args.secondary else [args.workload]
    for name in names:
        w = workloads.BY_NAME[name]
        line = measure(w, args, world, rank, local, want_e2e=not args.no_e2e and not args.secondary,
                       want_cpu=not args.no_cpu_baseline)
        if rank == 0:
            print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
