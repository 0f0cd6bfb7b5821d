"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each check is a hand-worked
value, a special case with a textbook form, a closed form, the pages'
chunked/segmented decomposition, finite differences, or an identity.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_inputs(seed, B, H, T, dk, dv, g_scale=0.3, s0=True):
    r = _rng(seed)
    q = r.standard_normal((B, H, T, dk))
    k = r.standard_normal((B, H, T, dk))
    v = r.standard_normal((B, H, T, dv))
    g = -np.abs(r.standard_normal((B, H, T, dk))) * g_scale
    S0 = r.standard_normal((B, H, dk, dv)) if s0 else None
    do = r.standard_normal((B, H, T, dv))
    dSf = r.standard_normal((B, H, dk, dv))
    return q, k, v, g, S0, do, dSf


def _read_golden(name):
    cases, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = cases.setdefault(vals[0], {})
                continue
            if cur is None:
                cur = cases.setdefault("", {})
            cur[key] = np.array([float(x) for x in vals])
    return cases


# ------------------------------------------------------------ hand-worked


def test_hand_scalar_case():
    cases = _read_golden("hand_scalar.txt")
    shp = (1, 1, 3, 1)
    q = np.ones(shp)
    k = np.ones(shp)
    v = np.array([1.0, 2.0, 3.0]).reshape(shp)
    g = np.full(shp, math.log(0.5))
    do = np.ones(shp)
    dSf = np.zeros((1, 1, 1, 1))
    z = cases["zero_init"]
    o, sf = oracle.gla_fwd(q, k, v, g, None)
    np.testing.assert_allclose(o.ravel(), z["o"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sf.ravel(), z["S_final"], rtol=1e-13)
    gr = oracle.gla_bwd(q, k, v, g, None, do, dSf)
    for name in ("dq", "dk", "dv", "dlog_alpha", "dS0"):
        np.testing.assert_allclose(gr[name].ravel(), z[name], rtol=1e-13, atol=1e-13,
                                   err_msg=name)
    s4 = cases["s0_four"]
    o, sf = oracle.gla_fwd(q, k, v, g, np.full((1, 1, 1, 1), 4.0))
    np.testing.assert_allclose(o.ravel(), s4["o"], rtol=1e-13)
    np.testing.assert_allclose(sf.ravel(), s4["S_final"], rtol=1e-13)


def test_hand_2x2_case():
    c = _read_golden("hand_2x2.txt")[""]
    T, dk, dv = 2, 2, 2
    q = c["q"].reshape(1, 1, T, dk)
    k = c["k"].reshape(1, 1, T, dk)
    v = c["v"].reshape(1, 1, T, dv)
    g = np.log(np.tile(c["alpha"], (T, 1))).reshape(1, 1, T, dk)
    do = c["do"].reshape(1, 1, T, dv)
    S0 = c["S0"].reshape(1, 1, dk, dv)
    dSf = c["dS_final"].reshape(1, 1, dk, dv)
    o, sf = oracle.gla_fwd(q, k, v, g, S0)
    np.testing.assert_allclose(o.ravel(), c["o"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sf.ravel(), c["S_final"], rtol=1e-13, atol=1e-13)
    gr = oracle.gla_bwd(q, k, v, g, S0, do, dSf)
    for name in ("dq", "dk", "dv", "dlog_alpha", "dS0"):
        np.testing.assert_allclose(gr[name].ravel(), c[name], rtol=1e-13, atol=1e-13,
                                   err_msg=name)


# --------------------------------------------- alpha == 1: causal attention


def test_alpha_one_is_causal_linear_attention():
    """With no decay the operator is causal (Q K^T * M) V plus the S0 term.

    The linear-attention left product inside a chunk and right product across
    chunks compute this same quantity (Linear Attention Sequence Parallelism,
    summary); here it is formed directly in O(T^2).
    """
    B, H, T, dk, dv = 1, 2, 160, 5, 7
    q, k, v, _, S0, do, dSf = _rand_inputs(1, B, H, T, dk, dv)
    g = np.zeros((B, H, T, dk))
    o, sf = oracle.gla_fwd(q, k, v, g, S0)
    gr = oracle.gla_bwd(q, k, v, g, S0, do, dSf)
    M = np.tril(np.ones((T, T)))
    for b in range(B):
        for h in range(H):
            Q, K_, V, dO = q[b, h], k[b, h], v[b, h], do[b, h]
            A = (Q @ K_.T) * M
            ref_o = A @ V + Q @ S0[b, h]
            ref_sf = S0[b, h] + K_.T @ V
            dA = (dO @ V.T) * M
            ref_dq = dA @ K_ + dO @ S0[b, h].T
            ref_dk = dA.T @ Q + V @ dSf[b, h].T
            ref_dv = A.T @ dO + K_ @ dSf[b, h]
            ref_dS0 = Q.T @ dO + dSf[b, h]
            np.testing.assert_allclose(o[b, h], ref_o, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(sf[b, h], ref_sf, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(gr["dq"][b, h], ref_dq, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(gr["dk"][b, h], ref_dk, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(gr["dv"][b, h], ref_dv, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(gr["dS0"][b, h], ref_dS0, rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------ closed form


def test_closed_form_constant_inputs_long_T():
    """Constant k, v and a constant per-row decay c_i give a geometric series:
    S_t[i,j] = c_i^(t+1) S0[i,j] + k_i v_j (1 - c_i^(t+1)) / (1 - c_i)."""
    T, dk, dv = 100_000, 3, 2
    c = np.array([0.9999, 0.99, 0.5])
    kv = np.array([0.7, -1.3, 2.0])
    vv = np.array([1.5, -0.25])
    qv = np.array([0.3, 0.2, -0.1])
    shp = (1, 1, T)
    q = np.broadcast_to(qv, shp + (dk,)).copy()
    k = np.broadcast_to(kv, shp + (dk,)).copy()
    v = np.broadcast_to(vv, shp + (dv,)).copy()
    g = np.broadcast_to(np.log(c), shp + (dk,)).copy()
    S0 = np.array([[1.0, -2.0], [0.5, 0.0], [3.0, 1.0]]).reshape(1, 1, dk, dv)
    o, sf = oracle.gla_fwd(q, k, v, g, S0)

    def S_at(n):  # state after n tokens
        cn = c ** n
        return cn[:, None] * S0[0, 0] + np.outer(kv * (1 - cn) / (1 - c), vv)

    np.testing.assert_allclose(sf[0, 0], S_at(T), rtol=1e-9)
    for t in (0, 1, 17, 999, 54321, T - 1):
        np.testing.assert_allclose(o[0, 0, t], qv @ S_at(t + 1), rtol=1e-9, atol=1e-12)


# ------------------------------------------- chunked / segmented form


@pytest.mark.parametrize("P,K,C", [(1, 1, 16), (4, 2, 16), (8, 3, 8), (32, 1, 8), (2, 6, 64),
                                   (16, 3, 4)])
def test_recurrence_equals_segmented_chunked_form(P, K, C):
    """Token recurrence == pass 1 + All-Scan + pass 2 for any P, K, C."""
    B, H, T, dk, dv = 2, 1, 256, 6, 5
    q, k, v, g, S0, _, _ = _rand_inputs(2, B, H, T, dk, dv, g_scale=0.2)
    if C >= T // P:
        C = T // P
    o_ref, sf_ref, S_in = chunked.chunked_fwd(q, k, v, g, S0, P, K, C)
    o, sf = oracle.gla_fwd(q, k, v, g, S0)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(sf, sf_ref, rtol=1e-11, atol=1e-11)
    # the segment-boundary states are the recurrence's states at t = pL - 1
    bs = oracle.boundary_states(q, k, v, g, S0, P)
    np.testing.assert_allclose(bs, S_in, rtol=1e-11, atol=1e-11)


# ------------------------------------------------- finite differences


def _loss(q, k, v, g, S0, do, dSf):
    o, sf = oracle.gla_fwd(q, k, v, g, S0, nthreads=1)
    return float(np.sum(o * do) + np.sum(sf * dSf))


def test_gradients_match_central_differences():
    B, H, T, dk, dv = 1, 2, 12, 3, 4
    q, k, v, g, S0, do, dSf = _rand_inputs(3, B, H, T, dk, dv)
    gr = oracle.gla_bwd(q, k, v, g, S0, do, dSf)
    h = 1e-6
    inputs = dict(q=q, k=k, v=v, g=g, S0=S0)
    names = dict(q="dq", k="dk", v="dv", g="dlog_alpha", S0="dS0")
    for nm, arr in inputs.items():
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(**inputs, do=do, dSf=dSf)
            arr[idx] = old - h
            lm = _loss(**inputs, do=do, dSf=dSf)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        an = gr[names[nm]]
        scale = max(1.0, np.abs(an).max())
        assert np.abs(fd - an).max() <= 1e-7 * scale, nm


def test_gradients_across_checkpoint_blocks():
    """T spans three checkpoint blocks of the backward (1024 tokens each)."""
    B, H, T, dk, dv = 1, 1, 2100, 2, 3
    q, k, v, g, S0, do, dSf = _rand_inputs(4, B, H, T, dk, dv, g_scale=0.002)
    gr = oracle.gla_bwd(q, k, v, g, S0, do, dSf)
    h = 1e-6
    r = _rng(5)
    inputs = dict(q=q, k=k, v=v, g=g)
    names = dict(q="dq", k="dk", v="dv", g="dlog_alpha")
    for nm, arr in inputs.items():
        for t in list(r.integers(0, T, 6)) + [0, 1023, 1024, 2047, 2048, T - 1]:
            d = int(r.integers(0, arr.shape[-1]))
            idx = (0, 0, int(t), d)
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(**inputs, S0=S0, do=do, dSf=dSf)
            arr[idx] = old - h
            lm = _loss(**inputs, S0=S0, do=do, dSf=dSf)
            arr[idx] = old
            fd = (lp - lm) / (2 * h)
            an = gr[names[nm]][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (nm, idx, fd, an)


# ------------------------------------------------------------ identities


def test_dlog_alpha_identity():
    """dg_t = sum_{s>=t} (q_s*dq_s - k_s*dk_s) + rowsum(dS_final * S_final).

    Scaling q_s[i] by e^eps and k_s[i] by e^-eps for all s >= t (and the
    final-state row by e^eps) is the same as shifting log_alpha_t[i] by eps;
    differentiating at eps = 0 gives the identity.
    """
    B, H, T, dk, dv = 2, 1, 90, 4, 3
    q, k, v, g, S0, do, dSf = _rand_inputs(6, B, H, T, dk, dv)
    _, sf = oracle.gla_fwd(q, k, v, g, S0)
    gr = oracle.gla_bwd(q, k, v, g, S0, do, dSf)
    term = q * gr["dq"] - k * gr["dk"]
    suffix = np.flip(np.cumsum(np.flip(term, axis=2), axis=2), axis=2)
    const = np.sum(dSf * sf, axis=-1)[:, :, None, :]
    np.testing.assert_allclose(gr["dlog_alpha"], suffix + const, rtol=1e-10, atol=1e-10)


def test_column_and_row_sampling_is_exact():
    """Sampled columns / rows are bit-identical to the same entries of a full run."""
    B, H, T, dk, dv = 1, 2, 300, 6, 7
    q, k, v, g, S0, do, dSf = _rand_inputs(7, B, H, T, dk, dv)
    o, sf = oracle.gla_fwd(q, k, v, g, S0)
    cols = [6, 0, 3]
    o_s, sf_s = oracle.gla_fwd(q, k, v, g, S0, cols=cols)
    assert np.array_equal(o_s, o[..., cols]) and np.array_equal(sf_s, sf[..., cols])
    full = oracle.gla_bwd(q, k, v, g, S0, do, dSf)
    rows = [5, 1]
    part = oracle.gla_bwd(q, k, v, g, S0, do, dSf, rows=rows, cols=cols)
    for nm in ("dq", "dk", "dlog_alpha"):
        assert np.array_equal(part[nm], full[nm][..., rows])
    assert np.array_equal(part["dS0"], full["dS0"][:, :, rows])
    assert np.array_equal(part["dv"], full["dv"][..., cols])


def test_empty_sequence():
    """T = 0: no outputs, S_final = S0, dS0 = dS_final."""
    q = np.zeros((1, 1, 0, 3))
    v = np.zeros((1, 1, 0, 2))
    S0 = np.arange(6.0).reshape(1, 1, 3, 2)
    dSf = -np.arange(6.0).reshape(1, 1, 3, 2)
    o, sf = oracle.gla_fwd(q, q, v, q, S0)
    assert o.shape == (1, 1, 0, 2) and np.array_equal(sf, S0)
    gr = oracle.gla_bwd(q, q, v, q, S0, v, dSf)
    assert np.array_equal(gr["dS0"], dSf)


def test_boundary_state_columns_match_full_states():
    B, H, T, dk, dv, P = 1, 2, 240, 4, 6, 5
    q, k, v, g, S0, _, _ = _rand_inputs(8, B, H, T, dk, dv)
    full = oracle.boundary_states(q, k, v, g, S0, P)
    cols = [5, 2]
    part = oracle.boundary_states_cols(q, k, v, g, S0, P, cols)
    np.testing.assert_allclose(part, full[..., cols], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------ other decay forms


def test_constant_scalar_decay_is_exponentially_weighted_causal_attention():
    # alpha_t = e^c for every token and every d_k row: S_t = sum_{s<=t} e^{c (t-s)} k_s^T v_s
    # (+ e^{c (t+1)} S0), so o = ((Q K^T) .* D) V + (e^{c (t+1)} q_t) S0 with
    # D[t, s] = e^{c (t - s)} for s <= t and 0 above the diagonal.
    B, H, T, dk, dv = 1, 2, 40, 5, 3
    q, k, v, _, S0, _, _ = _rand_inputs(11, B, H, T, dk, dv)
    c = -0.07
    g = np.full((B, H, T), c)
    o, sf = oracle.gla_fwd_decay(q, k, v, g, S0, oracle.DECAY_SCALAR)
    t = np.arange(T)
    D = np.where(t[:, None] >= t[None, :], np.exp(c * (t[:, None] - t[None, :])), 0.0)
    for b in range(B):
        for h in range(H):
            ref = ((q[b, h] @ k[b, h].T) * D) @ v[b, h]
            ref += (np.exp(c * (t + 1))[:, None] * q[b, h]) @ S0[b, h]
            assert np.abs(o[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
            sref = (np.exp(c * (T - 1 - t))[:, None] * k[b, h]).T @ v[b, h] + np.exp(c * T) * S0[b, h]
            assert np.abs(sf[b, h] - sref).max() <= 1e-12 * max(1.0, np.abs(sref).max())


def test_no_decay_is_causal_linear_attention():
    B, H, T, dk, dv = 1, 1, 30, 4, 6
    q, k, v, _, S0, _, _ = _rand_inputs(12, B, H, T, dk, dv)
    o, sf = oracle.gla_fwd_decay(q, k, v, None, S0, oracle.DECAY_NONE)
    M = np.tril(np.ones((T, T)))
    ref = ((q[0, 0] @ k[0, 0].T) * M) @ v[0, 0] + q[0, 0] @ S0[0, 0]
    assert np.abs(o[0, 0] - ref).max() <= 1e-12 * np.abs(ref).max()
    assert np.abs(sf[0, 0] - (k[0, 0].T @ v[0, 0] + S0[0, 0])).max() <= 1e-12 * 10


def test_scalar_decay_gradient_matches_central_differences():
    B, H, T, dk, dv = 1, 2, 10, 3, 4
    q, k, v, _, S0, do, dSf = _rand_inputs(13, B, H, T, dk, dv)
    g = -np.abs(_rng(14).standard_normal((B, H, T))) * 0.3
    gr = oracle.gla_bwd_decay(q, k, v, g, S0, do, dSf, oracle.DECAY_SCALAR)
    assert gr["dlog_alpha"].shape == (B, H, T)

    def loss(gs):
        o, sf = oracle.gla_fwd_decay(q, k, v, gs, S0, oracle.DECAY_SCALAR, nthreads=1)
        return float(np.sum(o * do) + np.sum(sf * dSf))

    h = 1e-6
    fd = np.zeros_like(g)
    for idx in np.ndindex(*g.shape):
        old = g[idx]
        g[idx] = old + h
        lp = loss(g)
        g[idx] = old - h
        lm = loss(g)
        g[idx] = old
        fd[idx] = (lp - lm) / (2 * h)
    scale = max(1.0, np.abs(gr["dlog_alpha"]).max())
    assert np.abs(fd - gr["dlog_alpha"]).max() <= 1e-7 * scale
    # the other gradients are those of the broadcast diagonal decay
    full = oracle.gla_bwd(q, k, v, np.repeat(g[..., None], dk, axis=-1), S0, do, dSf)
    for n in ("dq", "dk", "dv", "dS0"):
        assert np.array_equal(gr[n], full[n]), n
