"""Segmented, chunked fp64 evaluation of GLA, written from the ZeCO pages.

TEST INFRASTRUCTURE ONLY.  Its one job is to pin the token recurrence in
``oracle.c`` against the decomposition that the pages describe: the two
must agree to rounding (1e-11) for every choice of P, K and C.  It is plain
numpy, fp64, slow, and shares nothing with the CUDA library.

The steps, in the pages' order (ZeCO two-pass operator, Algorithm 1):

1. Pass 1 -- every segment p (tokens [pL, (p+1)L)) computes its local state
   from a zero state, chunk by chunk (Pith review of ZeCO, assumptions:
   Appendix A.1 -- the local recurrence can start from zero and be corrected
   later by the cumulative decay).  It also forms the segment's cumulative
   decay gamma[p] = prod_t alpha_t (per d_k row).
2. All-Scan -- the state is cut into K contiguous blocks of d_k rows; for
   every block, S_in[p+1] = (gamma[p]^T 1) * S_in[p] + S_loc[p]  (Pith review
   of ZeCO, "What carries the argument": the All-Scan update).  The state that
   travels on is the accumulated one (the pages' Algorithm 2 sends the local
   state in one branch; Pith review of ZeCO, referee major comment 4, calls
   that a bug, and the accumulated state is what the update defines).
3. Pass 2 -- every segment runs its chunks again from S_in[p]: outputs are the
   intra-chunk decay-masked attention plus the inter-chunk term q S, and the
   chunk state is carried.  Inside a chunk the decay between tokens s <= t is
   exp(b_t - b_s) with b the within-chunk inclusive cumulative log-decay; it
   is evaluated directly (never as a ratio of two exponentials).
"""
from __future__ import annotations

import numpy as np


def _chunk_terms(g_c):
    """Within-chunk cumulative log-decay b (inclusive) and its last row."""
    b = np.cumsum(g_c, axis=0)  # [C, dk]
    return b, b[-1]


def local_state(k_seg, v_seg, g_seg, C):
    """Pass 1 for one segment: state from zero plus gamma = exp(sum g)."""
    L, dk = k_seg.shape
    dv = v_seg.shape[1]
    S = np.zeros((dk, dv))
    for c0 in range(0, L, C):
        kc, vc, gc = k_seg[c0:c0 + C], v_seg[c0:c0 + C], g_seg[c0:c0 + C]
        b, blast = _chunk_terms(gc)
        khat = kc * np.exp(blast[None, :] - b)  # decay from token s to the chunk end
        S = np.exp(blast)[:, None] * S + khat.T @ vc
    gamma = np.exp(g_seg.sum(axis=0))
    return S, gamma


def all_scan(S0, S_loc, gamma, K):
    """Segment scan, block by block along d_k.  Returns S_in [P+1, dk, dv]."""
    P, dk, dv = S_loc.shape
    assert dk % K == 0
    blk = dk // K
    S_in = np.zeros((P + 1, dk, dv))
    S_in[0] = S0
    for kb in range(K):
        r = slice(kb * blk, (kb + 1) * blk)
        recv = S0[r]
        for p in range(P):
            send = gamma[p][r][:, None] * recv + S_loc[p][r]
            S_in[p + 1][r] = send
            recv = send  # forward the accumulated block, not the local one
    return S_in


def segment_outputs(q_seg, k_seg, v_seg, g_seg, S_start, C):
    """Pass 2 for one segment from its incoming global state."""
    L, dk = q_seg.shape
    dv = v_seg.shape[1]
    o = np.zeros((L, dv))
    S = S_start.copy()
    for c0 in range(0, L, C):
        qc, kc, vc, gc = q_seg[c0:c0 + C], k_seg[c0:c0 + C], v_seg[c0:c0 + C], g_seg[c0:c0 + C]
        n = qc.shape[0]
        b, blast = _chunk_terms(gc)
        # inter-chunk: (q_t * exp(b_t)) S
        o_inter = (qc * np.exp(b)) @ S
        # intra-chunk: A[t,s] = sum_i q_t[i] k_s[i] exp(b_t[i]-b_s[i]) for s <= t
        A = np.zeros((n, n))
        for t in range(n):
            for s in range(t + 1):
                A[t, s] = np.sum(qc[t] * kc[s] * np.exp(b[t] - b[s]))
        o[c0:c0 + n] = o_inter + A @ vc
        khat = kc * np.exp(blast[None, :] - b)
        S = np.exp(blast)[:, None] * S + khat.T @ vc
    return o


def chunked_fwd(q, k, v, g, S0, P, K, C):
    """Whole operator.  Arrays [B,H,T,D] (fp64); returns (o, S_final, S_in)."""
    q, k, v, g = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    assert T % P == 0
    L = T // P
    assert L % C == 0 or C >= L
    if S0 is None:
        S0 = np.zeros((B, H, dk, dv))
    S0 = np.asarray(S0, dtype=np.float64)
    o = np.zeros((B, H, T, dv))
    S_in_all = np.zeros((B, H, P + 1, dk, dv))
    for b_ in range(B):
        for h in range(H):
            S_loc = np.zeros((P, dk, dv))
            gam = np.zeros((P, dk))
            for p in range(P):
                sl = slice(p * L, (p + 1) * L)
                S_loc[p], gam[p] = local_state(k[b_, h, sl], v[b_, h, sl], g[b_, h, sl], C)
            S_in = all_scan(S0[b_, h], S_loc, gam, K)
            S_in_all[b_, h] = S_in
            for p in range(P):
                sl = slice(p * L, (p + 1) * L)
                o[b_, h, sl] = segment_outputs(q[b_, h, sl], k[b_, h, sl], v[b_, h, sl],
                                               g[b_, h, sl], S_in[p], C)
    return o, S_in_all[:, :, P], S_in_all
