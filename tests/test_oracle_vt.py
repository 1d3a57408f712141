"""Pins of the value-side transport oracle (CPU, fp64).

"Resumo Técnico: Por que Transformações Acumuladas Extrapolam?", §"Metodologia" 1 defines the route
transport P_{j->i} as the product of the per-token steps from source j to query i, and §"Principais
Contribuições" 3 "Proteção do Lado de Valor" applies the same accumulated transport to the values.
With PaTH's steps H_s = I - beta_s w_s w_s^T ("Resumo Técnico: Atenção PaTH", §2 "Mecanismo Central")
the operator that carries key j to query i in the logit is H_i ... H_{j+1}, so

    o_i = sum_j softmax_j(s_i.) H_i ... H_{j+1} v_j.

The oracle evaluates it left to right with one vector per row; the pins below fix it by explicit
d x d products, the beta = 0 library attention, closed forms, and decode-from-empty.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc


def _case(rng, L, d, beta_lo=0.0, beta_hi=2.0):
    q, k, v = (rng.standard_normal((L, d)) for _ in range(3))
    w = rng.standard_normal((L, d))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = rng.uniform(beta_lo, beta_hi, L)
    return q, k, v, w, beta


def _H(w, b):
    return np.eye(w.size) - b * np.outer(w, w)


def _dense_vt(q, k, v, w, beta, scale, order="route", log_f=None):
    """Explicit matrices: P_{j->i} = H_i ... H_{j+1} (route order), logits s_ij = scale q_i . P_{j->i} k_j
    (+ FoX bias), o_i = sum_j alpha_ij P_{j->i} v_j.  order='reversed' applies H_{j+1} ... H_i instead."""
    L, d = q.shape
    o, lse = np.zeros((L, d)), np.zeros(L)
    c = np.concatenate([[0.0], np.cumsum(log_f)]) if log_f is not None else None
    for i in range(L):
        Ps = []
        for j in range(i + 1):
            P = np.eye(d)
            steps = range(j + 1, i + 1)
            for s in steps:  # route order: H_{j+1} first, H_i last (leftmost)
                P = (_H(w[s], beta[s]) @ P) if order == "route" else (P @ _H(w[s], beta[s]))
            Ps.append(P)
        s = np.array([scale * q[i] @ Ps[j] @ k[j] for j in range(i + 1)])
        if c is not None:
            s = s + np.array([c[i + 1] - c[j + 1] for j in range(i + 1)])
        m = s.max()
        a = np.exp(s - m)
        lse[i] = m + np.log(a.sum())
        a /= a.sum()
        o[i] = sum(a[j] * (Ps[j] @ v[j]) for j in range(i + 1))
    return o, lse


@pytest.mark.parametrize("L,d,fox", [(7, 3, False), (12, 5, True), (16, 8, False)])
def test_vt_equals_explicit_route_products(L, d, fox):
    rng = np.random.default_rng(100 + L)
    q, k, v, w, beta = _case(rng, L, d)
    beta[2], beta[-1] = 0.0, 2.0
    lf = -rng.uniform(0.0, 1.0, L) if fox else None
    o_ref, lse_ref = _dense_vt(q, k, v, w, beta, 0.4, log_f=lf)
    o, lse = orc.path_attn(q, k, v, w, beta, log_f=lf, scale=0.4, value_transport=True)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    # the pin tells the route order from the reversed one and from untransported values
    o_rev, _ = _dense_vt(q, k, v, w, beta, 0.4, order="reversed", log_f=lf)
    o_plain, _ = orc.path_attn(q, k, v, w, beta, log_f=lf, scale=0.4)
    assert np.abs(o_rev - o).max() > 1e-3
    assert np.abs(o_plain - o).max() > 1e-3


def test_vt_logits_are_the_plain_ones():
    """Value transport changes the values only: lse equals the plain forward's."""
    rng = np.random.default_rng(5)
    q, k, v, w, beta = _case(rng, 40, 6)
    _, l1 = orc.path_attn(q, k, v, w, beta, scale=0.3, value_transport=True)
    _, l2 = orc.path_attn(q, k, v, w, beta, scale=0.3)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_vt_beta_zero_is_library_attention():
    rng = np.random.default_rng(6)
    q, k, v, w, beta = _case(rng, 50, 8)
    beta[:] = 0.0
    o, _ = orc.path_attn(q, k, v, w, beta, scale=0.35, value_transport=True)
    ref = torch.nn.functional.scaled_dot_product_attention(*(torch.from_numpy(x)[None] for x in (q, k, v)),
                                                           is_causal=True, scale=0.35)[0].numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_vt_d1_closed_form():
    """d = 1, w = +-1: every step multiplies by (1 - beta_s), so
    s_ij = scale q_i k_j prod_{s=j+1..i}(1 - beta_s) and o_i = sum_j alpha_ij v_j prod_{s=j+1..i}(1 - beta_s)."""
    rng = np.random.default_rng(7)
    L = 30
    q, k, v = (rng.standard_normal((L, 1)) for _ in range(3))
    w = np.where(rng.random((L, 1)) < 0.5, -1.0, 1.0)
    beta = rng.uniform(0, 2, L)
    o, _ = orc.path_attn(q, k, v, w, beta, scale=0.7, value_transport=True)
    for i in range(L):
        g = np.array([np.prod(1.0 - beta[j + 1:i + 1]) for j in range(i + 1)])
        s = 0.7 * q[i, 0] * k[:i + 1, 0] * g
        a = np.exp(s - s.max())
        a /= a.sum()
        assert abs(o[i, 0] - np.sum(a * v[:i + 1, 0] * g)) < 1e-12


def test_vt_constant_reflection_alternates():
    """Constant unit w with beta = 2: each step is the same reflection R (R^2 = I), so the route
    operator is R^((i - j) mod 2) and o_i = sum_j alpha_ij R^((i - j) mod 2) v_j."""
    rng = np.random.default_rng(8)
    L, d = 20, 5
    q, k, v, _, _ = _case(rng, L, d)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    w = np.tile(u, (L, 1))
    beta = np.full(L, 2.0)
    R = np.eye(d) - 2.0 * np.outer(u, u)
    o, _ = orc.path_attn(q, k, v, w, beta, scale=0.5, value_transport=True)
    for i in range(L):
        Ps = [np.linalg.matrix_power(R, (i - j) % 2) for j in range(i + 1)]
        s = np.array([0.5 * q[i] @ Ps[j] @ k[j] for j in range(i + 1)])
        a = np.exp(s - s.max())
        a /= a.sum()
        np.testing.assert_allclose(o[i], sum(a[j] * Ps[j] @ v[j] for j in range(i + 1)), rtol=0, atol=1e-12)


def test_vt_decode_from_empty_equals_forward():
    """Decoding with both caches transported in place (the values carried along the same route as
    the keys, §3 "Inferência" of the PaTH page applied to the value cache) reproduces the forward."""
    rng = np.random.default_rng(9)
    L, d = 33, 6
    q, k, v, w, beta = _case(rng, L, d)
    o_f, lse_f = orc.path_attn(q, k, v, w, beta, scale=0.45, value_transport=True)
    o_d, lse_d, kc, vc = orc.path_decode(np.zeros((0, d)), np.zeros((0, d)), q, k, v, w, beta, 0.45,
                                         value_transport=True)
    np.testing.assert_allclose(o_d, o_f, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_d, lse_f, rtol=0, atol=1e-12)
    # the value cache then holds H_{L-1} ... H_{j+1} v_j, the same transport as the keys
    for j in (0, 7, L - 1):
        x = v[j].copy()
        for t in range(j + 1, L):
            x = _H(w[t], beta[t]) @ x
        np.testing.assert_allclose(vc[j], x, rtol=0, atol=1e-12)
