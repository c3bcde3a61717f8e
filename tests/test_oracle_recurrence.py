"""Pins of the oracle's gated delta rule (CPU only).

The update pinned here is the one the pages' kernels follow (FLA's fused sigmoid-gated
recurrence, "[GDN] Spec-decoding-aware attention kernel", Changes and the closing note on
the SSM path): per (token, v-head), g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b),
S_t = e^g S_{t-1} (I - beta k k^T) + beta v k^T, o_t = S_t q / sqrt(dk), with L2-normed q, k.

Pins: closed forms at gate values whose transcendental results are exact facts
(softplus(0) = ln 2, sigmoid(0) = 1/2, sigmoid(-inf) = 0, sigmoid(+inf) = 1), the zero-prior
single-token outer product, the literal (I - beta k k^T) matrix form, the chunkwise WY
(UT-transform) form of the same recurrence (Yang et al., "Parallelizing Linear Transformers
with the Delta Rule over Sequence Length", 2024; Yang, Kautz & Hatamizadeh, "Gated Delta
Networks", 2025), the grouping of v-heads onto k-heads, and torch's own bf16 rounding.
"""
import math

import numpy as np
import pytest
import torch

import oracle

EPS = 1e-6


def _layer(Hk=2, Hv=4, dk=16, dv=16, bf16=False):
    return oracle.Layer(Hk, Hv, dk, dv, 4, 3, bf16)


def _rows_non_spec(lengths, slots, has_init=None):
    qsl = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    hi = None if has_init is None else np.asarray(has_init, np.int32)
    return oracle.Rows(qsl, False, None, np.asarray(slots, np.int32), hi)


def _rows_spec(lengths, ssi, num_acc):
    qsl = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return oracle.Rows(qsl, True, None, None, None, np.asarray(ssi, np.int32), np.asarray(num_acc, np.int32))


def _run(layer, qkv, a, b, A_log, dt, pool, rows):
    T = qkv.shape[0]
    out = np.zeros((T, layer.num_v_heads, layer.head_v_dim), np.float32)
    of = np.full(out.shape, np.nan)
    oracle.recurrent(layer, A_log.astype(np.float32), dt.astype(np.float32), pool, qkv, a, b, T, rows, out, of)
    return out, of


def _normed(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + EPS)


def _split(layer, qkv):
    Hk, Hv, dk, dv = layer.num_k_heads, layer.num_v_heads, layer.head_k_dim, layer.head_v_dim
    T = qkv.shape[0]
    q = qkv[:, : Hk * dk].reshape(T, Hk, dk)
    k = qkv[:, Hk * dk: 2 * Hk * dk].reshape(T, Hk, dk)
    v = qkv[:, 2 * Hk * dk:].reshape(T, Hv, dv)
    return q, k, v


def test_zero_prior_single_token_is_outer_product():
    L = _layer()
    rng = np.random.default_rng(0)
    qkv = rng.standard_normal((1, L.channels))
    a = rng.standard_normal((1, 4)).astype(np.float32)
    b = rng.standard_normal((1, 4)).astype(np.float32)
    pool = rng.standard_normal((3, 4, 16, 16)).astype(np.float32)
    out, of = _run(L, qkv, a, b, np.zeros(4), np.zeros(4), pool, _rows_non_spec([1], [2], [0]))
    q, k, v = _split(L, qkv)
    for h in range(4):
        kh = _normed(k[0, h // 2]); qh = _normed(q[0, h // 2]) / math.sqrt(16)
        beta = 1.0 / (1.0 + math.exp(-float(b[0, h])))
        S = beta * np.outer(v[0, h], kh)
        np.testing.assert_allclose(pool[2, h], S.astype(np.float32), rtol=1e-6, atol=1e-7)
        np.testing.assert_allclose(of[0, h], beta * v[0, h] * (kh @ qh), rtol=1e-12, atol=1e-14)


def test_beta_zero_is_pure_decay_by_half():
    """b = -inf gives beta = 0; A_log = 0 and a = -dt_bias give g = -ln 2, so each token halves S."""
    L = _layer()
    rng = np.random.default_rng(1)
    T = 3
    qkv = rng.standard_normal((T, L.channels))
    dt = rng.standard_normal(4).astype(np.float32)
    a = np.tile(-dt, (T, 1)).astype(np.float32)
    b = np.full((T, 4), -np.inf, np.float32)
    pool = rng.standard_normal((4, 4, 16, 16)).astype(np.float32)
    S0 = pool[1].astype(np.float64).copy()
    out, of = _run(L, qkv, a, b, np.zeros(4), dt, pool, _rows_non_spec([T], [1]))
    np.testing.assert_allclose(pool[1], (S0 / 2 ** T).astype(np.float32), rtol=1e-7, atol=0)
    q, _, _ = _split(L, qkv)
    for t in range(T):
        for h in range(4):
            qh = _normed(q[t, h // 2]) / 4.0
            np.testing.assert_allclose(of[t, h], (S0[h] / 2 ** (t + 1)) @ qh, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("b_val", [0.0, np.inf])
def test_one_step_key_identity(b_val):
    """S_t k_t = e^g (1 - beta|k|^2) S_{t-1} k_t + beta |k|^2 v_t (here e^g = 1/2, beta = 1/2 or 1)."""
    L = _layer()
    rng = np.random.default_rng(2)
    qkv = rng.standard_normal((1, L.channels))
    dt = rng.standard_normal(4).astype(np.float32)
    a = (-dt)[None].astype(np.float32)
    b = np.full((1, 4), b_val, np.float32)
    beta = 0.5 if b_val == 0.0 else 1.0
    pool = rng.standard_normal((3, 4, 16, 16)).astype(np.float32)
    S0 = pool[1].astype(np.float64).copy()
    _run(L, qkv, a, b, np.zeros(4), dt, pool, _rows_non_spec([1], [1]))
    _, k, v = _split(L, qkv)
    for h in range(4):
        kh = _normed(k[0, h // 2])
        kk = kh @ kh
        expect = 0.5 * (1 - beta * kk) * (S0[h] @ kh) + beta * kk * v[0, h]
        np.testing.assert_allclose(pool[1, h].astype(np.float64) @ kh, expect, rtol=1e-5, atol=1e-5)


def _literal(layer, qkv, a, b, A_log, dt, S0, store_every=False):
    """S_t = e^g S (I - beta k k^T) + beta v k^T, o = S q, with explicit matrices."""
    q, k, v = _split(layer, qkv)
    Hv, dk = layer.num_v_heads, layer.head_k_dim
    G = Hv // layer.num_k_heads
    S = S0.astype(np.float64).copy()
    outs, states = [], []
    for t in range(qkv.shape[0]):
        o = np.zeros((Hv, layer.head_v_dim))
        for h in range(Hv):
            kh = _normed(k[t, h // G]); qh = _normed(q[t, h // G]) / math.sqrt(dk)
            g = -math.exp(float(A_log[h])) * math.log1p(math.exp(float(a[t, h]) + float(dt[h])))
            beta = 1.0 / (1.0 + math.exp(-float(b[t, h])))
            S[h] = math.exp(g) * S[h] @ (np.eye(dk) - beta * np.outer(kh, kh)) + beta * np.outer(v[t, h], kh)
            o[h] = S[h] @ qh
        outs.append(o)
        states.append(S.copy())
    return np.stack(outs), states


def test_literal_matrix_form_spec_row():
    L = _layer(Hk=2, Hv=4, dk=8, dv=4)
    rng = np.random.default_rng(3)
    T = 4
    qkv = rng.standard_normal((T, L.channels))
    a = rng.standard_normal((T, 4)).astype(np.float32)
    b = rng.standard_normal((T, 4)).astype(np.float32)
    A_log = np.log(rng.uniform(1, 16, 4)).astype(np.float32)
    dt = (0.1 * rng.standard_normal(4)).astype(np.float32)
    pool = rng.standard_normal((10, 4, 4, 8)).astype(np.float32)
    ssi = np.array([[3, 7, 5, 9]], np.int32)
    S0 = pool[7].copy()  # num_accepted = 2 -> load column 1
    out, of = _run(L, qkv, a, b, A_log, dt, pool, _rows_spec([T], ssi, [2]))
    ref_o, ref_s = _literal(L, qkv, a, b, A_log, dt, S0)
    np.testing.assert_allclose(of, ref_o, rtol=1e-11, atol=1e-12)
    for t in range(T):
        np.testing.assert_allclose(pool[ssi[0, t]], ref_s[t].astype(np.float32), rtol=1e-6, atol=1e-7)


def _chunked(layer, qkv, a, b, A_log, dt, S0, c):
    """Chunkwise WY form of the same recurrence, float64, per v-head."""
    q, k, v = _split(layer, qkv)
    T = qkv.shape[0]
    Hv, dk = layer.num_v_heads, layer.head_k_dim
    G_ = Hv // layer.num_k_heads
    outs = np.zeros((T, Hv, layer.head_v_dim))
    S_fin = np.zeros_like(S0, dtype=np.float64)
    for h in range(Hv):
        Q = _normed(q[:, h // G_]) / math.sqrt(dk)
        K = _normed(k[:, h // G_])
        V = v[:, h]
        g = np.array([-math.exp(float(A_log[h])) * math.log1p(math.exp(float(a[t, h]) + float(dt[h])))
                      for t in range(T)])
        beta = 1.0 / (1.0 + np.exp(-b[:, h].astype(np.float64)))
        S = S0[h].astype(np.float64)
        for c0 in range(0, T, c):
            sl = slice(c0, min(T, c0 + c))
            Qc, Kc, Vc, Bc = Q[sl], K[sl], V[sl], beta[sl]
            Gc = np.cumsum(g[sl])
            n = len(Gc)
            D = Gc[:, None] - Gc[None, :]
            strict = np.tril(np.ones((n, n)), -1)
            incl = np.tril(np.ones((n, n)))
            A = strict * Bc[:, None] * np.exp(np.where(strict > 0, D, 0.0)) * (Kc @ Kc.T)
            Tm = np.linalg.inv(np.eye(n) + A)
            W = Tm @ (Bc[:, None] * np.exp(Gc)[:, None] * Kc)
            U = Tm @ (Bc[:, None] * Vc) - W @ S.T
            P = incl * np.exp(np.where(incl > 0, D, 0.0)) * (Qc @ Kc.T)
            outs[sl, h] = np.exp(Gc)[:, None] * (Qc @ S.T) + P @ U
            S = math.exp(Gc[-1]) * S + (U * np.exp(Gc[-1] - Gc)[:, None]).T @ Kc
        S_fin[h] = S
    return outs, S_fin


@pytest.mark.parametrize("T,c", [(77, 16), (64, 64), (5, 8)])
def test_chunked_wy_form_equals_token_recurrence(T, c):
    L = _layer(Hk=2, Hv=4, dk=16, dv=8)
    rng = np.random.default_rng(4 + T)
    qkv = rng.standard_normal((T, L.channels))
    a = rng.standard_normal((T, 4)).astype(np.float32)
    b = rng.standard_normal((T, 4)).astype(np.float32)
    A_log = np.log(rng.uniform(1, 16, 4)).astype(np.float32)
    dt = (0.1 * rng.standard_normal(4)).astype(np.float32)
    pool = rng.standard_normal((3, 4, 8, 16)).astype(np.float32)
    S0 = pool[2].copy()
    out, of = _run(L, qkv, a, b, A_log, dt, pool, _rows_non_spec([T], [2]))
    ref_o, ref_S = _chunked(L, qkv, a, b, A_log, dt, S0, c)
    np.testing.assert_allclose(of, ref_o, rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(pool[2], ref_S.astype(np.float32), rtol=1e-6, atol=1e-7)


def test_scalar_head_brute_force():
    """dk = dv = 1: k^ = k/sqrt(k^2+eps), and the update is a scalar recursion."""
    L = oracle.Layer(1, 1, 1, 1, 4, 3, False)
    rng = np.random.default_rng(5)
    T = 9
    qkv = rng.standard_normal((T, 3))
    a = rng.standard_normal((T, 1)).astype(np.float32)
    b = rng.standard_normal((T, 1)).astype(np.float32)
    A_log = np.array([0.7], np.float32); dt = np.array([0.05], np.float32)
    pool = np.array([0.0, 0.3, 0.0], np.float32).reshape(3, 1, 1, 1)
    s = float(pool[1, 0, 0, 0])
    out, of = _run(L, qkv, a, b, A_log, dt, pool, _rows_non_spec([T], [1]))
    for t in range(T):
        qn = qkv[t, 0] / math.sqrt(qkv[t, 0] ** 2 + EPS)
        kn = qkv[t, 1] / math.sqrt(qkv[t, 1] ** 2 + EPS)
        decay = math.exp(-math.exp(float(A_log[0])) * math.log1p(math.exp(float(a[t, 0]) + float(dt[0]))))
        beta = 1 / (1 + math.exp(-float(b[t, 0])))
        s = decay * s * (1 - beta * kn * kn) + beta * qkv[t, 2] * kn
        assert abs(of[t, 0, 0] - s * qn) <= 1e-13
    assert abs(pool[1, 0, 0, 0] - np.float32(s)) == 0


def test_v_heads_group_consecutively_onto_k_heads():
    """With every v-head given the same v, gates and prior, heads h and h' agree exactly iff
    they share the k-head h // (Hv/Hk)."""
    L = _layer(Hk=2, Hv=4, dk=8, dv=8)
    rng = np.random.default_rng(6)
    T = 3
    qkv = rng.standard_normal((T, L.channels))
    v = qkv[:, 2 * 16:].reshape(T, 4, 8)
    v[:] = v[:, :1]
    a = np.tile(rng.standard_normal((T, 1)), (1, 4)).astype(np.float32)
    b = np.tile(rng.standard_normal((T, 1)), (1, 4)).astype(np.float32)
    pool = np.tile(rng.standard_normal((3, 1, 8, 8)), (1, 4, 1, 1)).astype(np.float32)
    out, of = _run(L, qkv, a, b, np.full(4, 0.5), np.zeros(4), pool, _rows_non_spec([T], [1]))
    assert np.array_equal(of[:, 0], of[:, 1]) and np.array_equal(of[:, 2], of[:, 3])
    assert not np.allclose(of[:, 0], of[:, 2])


def test_bf16_outputs_round_like_torch():
    L = _layer(bf16=True)
    rng = np.random.default_rng(7)
    T = 6
    qkv = rng.standard_normal((T, L.channels))
    to_bits = lambda x: torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    a = to_bits(rng.standard_normal((T, 4)).astype(np.float32))
    b = to_bits(rng.standard_normal((T, 4)).astype(np.float32))
    pool = rng.standard_normal((3, 4, 16, 16)).astype(np.float32)
    out = np.zeros((T, 4, 16), np.uint16)
    of = np.zeros((T, 4, 16))
    oracle.recurrent(L, np.zeros(4, np.float32), np.zeros(4, np.float32), pool, qkv, a, b, T,
                     _rows_non_spec([T], [1]), out, of)
    expect = torch.from_numpy(of).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, expect)
