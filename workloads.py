"""Seeded synthetic workloads for segmented gated linear attention.

This module only draws random tensors and names shapes. It contains none of
the attention arithmetic, so the CPU oracle (``oracle/``) and the CUDA path
(``chunked_state_scan_gb300``) can both take their inputs from it without
sharing any of the method.

The shapes follow the GLA-1B attention layer that the ZeCO operator runs were
made on (ZeCO: Zero-Communication Overhead Sequence Parallelism for Linear
Attention, experimental setup: 16k tokens per device, state d_k x d_v), with
the per-head sizes d_k=256, d_v=512 and H=4 heads.  The pages measure on no
public dataset; every tensor here is synthetic.

Recipe (one generator, drawn in this order): q, k, v, x, do, dS_final, S0.
Each is drawn in fp32 and then cast to the I/O dtype.  The decay input is
``log_alpha = logsigmoid(x) / 16`` evaluated in fp32 and then cast, so that
both sides see exactly the same rounded values.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    P: int  # segments
    K: int  # d_k blocks of the segment scan
    C: int  # chunk length
    dtype: str  # "f32" or "bf16" (I/O dtype; accumulation is always fp32)
    seed: int
    qk_scale: float  # q, k ~ N(0,1) * qk_scale
    v_scale: float  # v ~ N(0,1) * v_scale
    x_mean: float  # log_alpha = logsigmoid(N(x_mean, 1)) / 16
    s0_scale: float  # S0 ~ N(0,1) * s0_scale (0 means S0 = 0)
    bwd: bool  # whether the workload includes the backward
    dsf_scale: float = 0.1  # dS_final ~ N(0,1) * dsf_scale

    @property
    def L(self) -> int:
        return self.T // self.P

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def replace(self, **kw) -> "Workload":
        d = asdict(self)
        d.update(kw)
        return Workload(**d)


# The five workloads, in order: the tiny fp32 case, the GLA-1B layer shape with
# one segment, the 8-segment forward, the 1M-token 64-segment forward+backward
# (the throughput workload) and the batched slow-decay forward+backward.
TINY_F32 = Workload("tiny_f32_T1024_P4", B=1, H=2, T=1024, dk=64, dv=64, P=4, K=2, C=64,
                    dtype="f32", seed=0, qk_scale=1 / 8, v_scale=1 / 8, x_mean=0.0,
                    s0_scale=0.0, bwd=False)
GLA1B_FWD = Workload("gla1b_fwd_T16384_P1", B=1, H=4, T=16384, dk=256, dv=512, P=1, K=1, C=64,
                     dtype="bf16", seed=1, qk_scale=1 / 16, v_scale=1.0, x_mean=0.0,
                     s0_scale=0.0, bwd=False)
SEG_FWD = Workload("seg_fwd_T131072_P8", B=1, H=4, T=131072, dk=256, dv=512, P=8, K=4, C=64,
                   dtype="bf16", seed=2, qk_scale=1 / 16, v_scale=1.0, x_mean=0.0,
                   s0_scale=0.0, bwd=False)
LONG_FWDBWD = Workload("long_fwdbwd_T1048576_P64", B=1, H=4, T=1048576, dk=256, dv=512, P=64,
                       K=8, C=64, dtype="bf16", seed=3, qk_scale=1 / 16, v_scale=1.0,
                       x_mean=0.0, s0_scale=0.0, bwd=True)
BATCHED_FWDBWD = Workload("batched_fwdbwd_B8_T32768_P2", B=8, H=4, T=32768, dk=256, dv=512,
                          P=2, K=4, C=64, dtype="bf16", seed=4, qk_scale=1 / 16, v_scale=1.0,
                          x_mean=2.0, s0_scale=0.1, bwd=True)

WORKLOADS = [TINY_F32, GLA1B_FWD, SEG_FWD, LONG_FWDBWD, BATCHED_FWDBWD]

# Small case of the throughput workload for ncu captures: the same kernels and
# shapes per token, 1/32 of the tokens (one wave of CTAs, inputs 470 MB > L2).
PROFILE_FWDBWD = LONG_FWDBWD.replace(name="profile_fwdbwd_T32768_P8", T=32768, P=8)

# The throughput workload cut into P = T/C segments of one chunk each: the segment
# scans (a long chain of 16,384 states per (b, h)) then take about as long as the
# rest of the step, the regime in which hiding them beside other work matters.
SCAN_BOUND_FWDBWD = LONG_FWDBWD.replace(name="long_fwdbwd_T1048576_P16384", P=16384)

# The throughput workload with small heads (d_k = 64, d_v = 128): the tensor-core
# kernels' partial tiles of 128 d_k rows and the native d_k = 64 sweeps.
SMALL_HEAD_FWDBWD = LONG_FWDBWD.replace(name="small_head_fwdbwd_T1048576_dk64_dv128", dk=64,
                                        dv=128, K=2)

BY_NAME = {w.name: w for w in WORKLOADS + [PROFILE_FWDBWD, SCAN_BOUND_FWDBWD,
                                            SMALL_HEAD_FWDBWD]}


def make_inputs(w: Workload, device="cpu", seed: int | None = None):
    """Draw the inputs of workload ``w`` on ``device``.

    Returns a dict of tensors: q, k, log_alpha [B,H,T,dk]; v, do [B,H,T,dv]
    in the I/O dtype; S0, dS_final [B,H,dk,dv] in fp32.
    """
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    dt = w.torch_dtype

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)

    q = (randn(B, H, T, dk) * w.qk_scale).to(dt)
    k = (randn(B, H, T, dk) * w.qk_scale).to(dt)
    v = (randn(B, H, T, dv) * w.v_scale).to(dt)
    x = randn(B, H, T, dk)
    if w.x_mean:
        x.add_(w.x_mean)
    log_alpha = (torch.nn.functional.logsigmoid(x) / 16.0).to(dt)
    del x
    do = randn(B, H, T, dv).to(dt)
    dS_final = randn(B, H, dk, dv) * w.dsf_scale
    if w.s0_scale:
        S0 = randn(B, H, dk, dv) * w.s0_scale
    else:
        S0 = torch.zeros(B, H, dk, dv, device=device, dtype=torch.float32)
    return dict(q=q, k=k, v=v, log_alpha=log_alpha, do=do, dS_final=dS_final, S0=S0)


def make_custom(B, H, T, dk, dv, dtype="f32", seed=0, qk_scale=None, v_scale=1.0, x_mean=0.0,
                x_scale=1.0, g_zero=False, s0_scale=0.0, device="cpu"):
    """Inputs of an arbitrary shape with the same recipe (used by edge-case tests).

    ``x_mean`` shifts the decay logits (large ``x_mean`` gives slow decay);
    ``g_zero`` sets log_alpha to exactly zero (no decay).
    """
    if qk_scale is None:
        qk_scale = 1.0 / math.sqrt(dk)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)

    q = (randn(B, H, T, dk) * qk_scale).to(dt)
    k = (randn(B, H, T, dk) * qk_scale).to(dt)
    v = (randn(B, H, T, dv) * v_scale).to(dt)
    x = randn(B, H, T, dk) * x_scale + x_mean
    if g_zero:
        log_alpha = torch.zeros(B, H, T, dk, device=device, dtype=dt)
    else:
        log_alpha = (torch.nn.functional.logsigmoid(x) / 16.0).to(dt)
    do = randn(B, H, T, dv).to(dt)
    dS_final = randn(B, H, dk, dv) * 0.1
    S0 = randn(B, H, dk, dv) * s0_scale if s0_scale else torch.zeros(B, H, dk, dv, device=device)
    return dict(q=q, k=k, v=v, log_alpha=log_alpha, do=do, dS_final=dS_final, S0=S0)
