"""Pins for the fp64 CPU oracle (CPU only).

Each test ties oracle/ to something other than itself: a hand-derived example,
a brute-force dense product, a library routine at a special case, a closed
form or an invariant.  Definitions follow "Resumo Técnico: Atenção PaTH"
(gist.science/pt/paper/2505.16381): §2 "Mecanismo Central" (logit and
transition equations), §2 "Extensões: PaTH-FoX", §3 "Representação de
Transformação UT" and §3 "Inferência".
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import dense
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, L, d, edge=True, unit=True):
    q, k, v = (rng.standard_normal((L, d)) for _ in range(3))
    w = rng.standard_normal((L, d))
    if unit:
        w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = 2.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    if edge and L > 2:
        beta[rng.integers(0, L)] = 0.0
        beta[rng.integers(0, L)] = 2.0
    return q, k, v, w, beta


def _softmax_rows(S, V):
    m = np.max(S, axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    return (P / l) @ V, (m + np.log(l))[:, 0]


# --------------------------------------------------------------------------- golden
def test_golden_hand_derived_logits():
    g = json.load(open(os.path.join(GOLDEN, "hand_d2_L3.json")))
    q, k, v, w, beta = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "v", "w", "beta"))
    S = orc.path_logits(q, k, w, beta, scale=1.0)
    exp = np.array([[np.nan if x is None else x for x in r] for r in g["logits"]])
    mask = ~np.isnan(exp)
    np.testing.assert_allclose(S[mask], exp[mask], rtol=0, atol=1e-12)
    assert np.all(np.isneginf(S[~mask]))
    # the descending product order gives a different (wrong) value
    assert abs(S[2, 0] - g["logit20_descending_order"]) > 1.0
    # o and lse from the golden logits, by hand
    o, lse = orc.path_attn(q, k, v, w, beta, scale=1.0)
    for i in range(3):
        s = [exp[i, j] for j in range(i + 1)]
        m = max(s)
        p = [math.exp(x - m) for x in s]
        l = sum(p)
        o_ref = [sum(p[j] * v[j, c] for j in range(i + 1)) / l for c in range(2)]
        assert np.allclose(o[i], o_ref, atol=1e-12)
        assert abs(lse[i] - (m + math.log(l))) < 1e-12


def test_golden_hand_derived_fox_logits():
    g = json.load(open(os.path.join(GOLDEN, "hand_d2_L3.json")))
    q, k, w, beta, lf = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "w", "beta", "log_f"))
    S = orc.path_logits(q, k, w, beta, log_f=lf, scale=1.0)
    exp = np.array([[np.nan if x is None else x for x in r] for r in g["logits_fox"]])
    mask = ~np.isnan(exp)
    np.testing.assert_allclose(S[mask], exp[mask], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- brute force
@pytest.mark.parametrize("L,d,seed", [(1, 3, 0), (2, 2, 1), (5, 1, 2), (9, 4, 3), (17, 8, 4), (24, 16, 5)])
def test_walk_matches_dense_product(L, d, seed):
    rng = np.random.default_rng(seed)
    q, k, v, w, beta = _rand_case(rng, L, d)
    scale = 1.0 / math.sqrt(d)
    S = orc.path_logits(q, k, w, beta, scale=scale)
    Sd = dense.logits(q, k, w, beta, scale=scale)
    tri = np.tril(np.ones((L, L), bool))
    np.testing.assert_allclose(S[tri], Sd[tri], rtol=0, atol=1e-12)
    o, lse = orc.path_attn(q, k, v, w, beta, scale=scale)
    od, lsed = dense.attention(q, k, v, w, beta, scale=scale)
    np.testing.assert_allclose(o, od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lsed, rtol=0, atol=1e-12)


def test_walk_matches_dense_product_fox():
    rng = np.random.default_rng(11)
    q, k, v, w, beta = _rand_case(rng, 13, 5)
    lf = np.log(1.0 / (1.0 + np.exp(-(3.0 + rng.standard_normal(13)))))
    o, lse = orc.path_attn(q, k, v, w, beta, log_f=lf, scale=0.5)
    od, lsed = dense.attention(q, k, v, w, beta, scale=0.5, log_f=lf)
    np.testing.assert_allclose(o, od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lsed, rtol=0, atol=1e-12)


def test_non_unit_w_used_as_given():
    """The oracle neither normalises w nor clips beta: a non-unit w must match the dense product."""
    rng = np.random.default_rng(3)
    q, k, v, w, beta = _rand_case(rng, 10, 4, unit=False)
    o, _ = orc.path_attn(q, k, v, w, beta, scale=1.0)
    od, _ = dense.attention(q, k, v, w, beta, scale=1.0)
    np.testing.assert_allclose(o, od, rtol=0, atol=1e-10)


# --------------------------------------------------------------------------- library special case
@pytest.mark.parametrize("L,d", [(64, 16), (33, 8)])
def test_beta_zero_is_causal_softmax_attention(L, d):
    """beta = 0 makes every H_s the identity: ordinary causal softmax attention (torch SDPA, fp64)."""
    rng = np.random.default_rng(5)
    q, k, v, w, _ = _rand_case(rng, L, d)
    beta = np.zeros(L)
    scale = 1.0 / math.sqrt(d)
    o, lse = orc.path_attn(q, k, v, w, beta, scale=scale)
    t = lambda a: torch.from_numpy(a)[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True, scale=scale)
    np.testing.assert_allclose(o, ref[0, 0].numpy(), rtol=0, atol=1e-12)
    S = scale * q @ k.T + np.triu(np.full((L, L), -np.inf), 1)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(S), dim=1).numpy(), atol=1e-12)


# --------------------------------------------------------------------------- closed forms
def test_d1_closed_form():
    """d = 1, w = +-1: H_s = 1 - beta_s, so s_ij = k_j q_i prod_{s=j+1}^{i} (1 - beta_s)."""
    rng = np.random.default_rng(7)
    L = 12
    q, k = rng.standard_normal((L, 1)), rng.standard_normal((L, 1))
    w = np.where(rng.random((L, 1)) < 0.5, -1.0, 1.0)
    beta = rng.random(L) * 2
    S = orc.path_logits(q, k, w, beta, scale=1.0)
    for i in range(L):
        for j in range(i + 1):
            prod = 1.0
            for s in range(j + 1, i + 1):
                prod *= 1.0 - beta[s]
            assert abs(S[i, j] - k[j, 0] * q[i, 0] * prod) < 1e-12


def test_constant_w_reflection_alternates():
    """Constant unit w and beta = 2: H is a reflection with H^2 = I, so the logit is
    k_j.q_i for even i - j and k_j.(H q_i) for odd i - j."""
    rng = np.random.default_rng(8)
    L, d = 11, 6
    q, k = rng.standard_normal((L, d)), rng.standard_normal((L, d))
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    w = np.tile(u, (L, 1))
    beta = np.full(L, 2.0)
    S = orc.path_logits(q, k, w, beta, scale=1.0)
    for i in range(L):
        Hq = q[i] - 2.0 * (u @ q[i]) * u
        for j in range(i + 1):
            ref = k[j] @ (q[i] if (i - j) % 2 == 0 else Hq)
            assert abs(S[i, j] - ref) < 1e-12


@pytest.mark.parametrize("beta_val,expect", [(2.0, "equal"), (1.0, "shrink")])
def test_reflection_product_preserves_norm(beta_val, expect):
    """beta = 2 with unit w makes each H_s a reflection, so prod H_s is orthogonal and
    |P q| = |q|.  Reading the transported query through basis keys k_j = e_c gives
    the components of P_{j->i} q_i one at a time.  beta = 1 (projectors) must shrink it."""
    rng = np.random.default_rng(9)
    L, d = 20, 5
    q = rng.standard_normal((L, d))
    w = rng.standard_normal((L, d))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = np.full(L, beta_val)
    comps = []
    for c in range(d):
        k = np.zeros((L, d))
        k[:, c] = 1.0
        comps.append(orc.path_logits(q, k, w, beta, scale=1.0))
    comps = np.stack(comps)  # [d, L, L]: comps[c, i, j] = (P_{j->i} q_i)_c
    for i in range(L):
        for j in range(i + 1):
            n = np.linalg.norm(comps[:, i, j])
            if expect == "equal":
                assert abs(n - np.linalg.norm(q[i])) < 1e-12
            elif j < i - 2:
                assert n < np.linalg.norm(q[i]) - 1e-9


# --------------------------------------------------------------------------- FoX special cases
def test_fox_with_beta_zero_is_additive_bias_attention():
    rng = np.random.default_rng(12)
    L, d = 40, 8
    q, k, v, w, _ = _rand_case(rng, L, d)
    beta = np.zeros(L)
    lf = np.log(1.0 / (1.0 + np.exp(-(3.0 + rng.standard_normal(L)))))
    o, lse = orc.path_attn(q, k, v, w, beta, log_f=lf, scale=0.3)
    S = np.full((L, L), -np.inf)
    for i in range(L):
        for j in range(i + 1):
            S[i, j] = 0.3 * (q[i] @ k[j]) + sum(lf[s] for s in range(j + 1, i + 1))
    o_ref, lse_ref = _softmax_rows(S, v)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_fox_with_zero_gates_equals_plain():
    rng = np.random.default_rng(13)
    q, k, v, w, beta = _rand_case(rng, 30, 6)
    o1, l1 = orc.path_attn(q, k, v, w, beta, log_f=np.zeros(30), scale=0.4)
    o2, l2 = orc.path_attn(q, k, v, w, beta, scale=0.4)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# --------------------------------------------------------------------------- UT transform reading
@pytest.mark.parametrize("C,d,seed", [(4, 3, 0), (16, 16, 1), (32, 16, 2), (64, 64, 3), (128, 128, 4), (128, 64, 5)])
def test_ut_identity(C, d, seed):
    """§3 "Representação de Transformação UT": the product of C transitions is I - W^T T^{-1} W
    with T triangular and built from beta.  Reading: T = diag(1/beta) + triu_1(W W^T) (ascending
    product), equivalently the division-free A = (I + D triu_1(W W^T))^{-1} D, exact at beta = 0.
    The GPU UT-prep kernel relies on this reading; here it is checked against the explicit product."""
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((C, d))
    W /= np.linalg.norm(W, axis=1, keepdims=True)
    beta = 2.0 / (1.0 + np.exp(-rng.standard_normal(C)))
    P = dense.path_product(np.vstack([np.zeros((1, d)), W]), np.concatenate([[0.0], beta]), 0, C)
    G = W @ W.T
    T = np.diag(1.0 / beta) + np.triu(G, 1)
    np.testing.assert_allclose(P, np.eye(d) - W.T @ np.linalg.solve(T, W), atol=1e-11)
    beta[0] = 0.0
    beta[-1] = 2.0
    P = dense.path_product(np.vstack([np.zeros((1, d)), W]), np.concatenate([[0.0], beta]), 0, C)
    D = np.diag(beta)
    A = np.linalg.solve(np.eye(C) + D @ np.triu(G, 1), D)
    assert np.allclose(A, np.triu(A))
    np.testing.assert_allclose(P, np.eye(d) - W.T @ A @ W, atol=1e-11)


# --------------------------------------------------------------------------- decode invariant
@pytest.mark.parametrize("L,d,seed", [(1, 4, 0), (7, 3, 1), (25, 8, 2)])
def test_decode_from_empty_cache_equals_prefill(L, d, seed):
    """§3 "Inferência": updating the cached keys in place with each step's transition and then
    attending with the plain query reproduces the prefill rows."""
    rng = np.random.default_rng(seed)
    q, k, v, w, beta = _rand_case(rng, L, d)
    o_pre, lse_pre = orc.path_attn(q, k, v, w, beta, scale=0.7)
    o_dec, lse_dec, _, _ = orc.path_decode(np.zeros((0, d)), np.zeros((0, d)), q, k, v, w, beta, 0.7)
    np.testing.assert_allclose(o_dec, o_pre, atol=1e-12)
    np.testing.assert_allclose(lse_dec, lse_pre, atol=1e-12)


def test_decode_after_prefilled_cache_equals_prefill():
    """A cache holding the dense-product transported keys H_{n0-1}...H_{j+1} k_j, continued by
    decode steps, gives the prefill rows of the whole sequence."""
    rng = np.random.default_rng(21)
    L, n0, d = 18, 11, 5
    q, k, v, w, beta = _rand_case(rng, L, d)
    kc0 = np.stack([dense.path_product(w, beta, j, n0 - 1).T @ k[j] for j in range(n0)])
    o_pre, _ = orc.path_attn(q, k, v, w, beta, scale=0.5)
    o_dec, _, kc, _ = orc.path_decode(kc0, v[:n0], q[n0:], k[n0:], v[n0:], w[n0:], beta[n0:], 0.5)
    np.testing.assert_allclose(o_dec, o_pre[n0:], atol=1e-12)
    kc_ref = np.stack([dense.path_product(w, beta, j, L - 1).T @ k[j] for j in range(L)])
    np.testing.assert_allclose(kc, kc_ref, atol=1e-12)


def test_kcache_update_is_one_transition():
    rng = np.random.default_rng(22)
    kc = rng.standard_normal((9, 6))
    w = rng.standard_normal(6)
    w /= np.linalg.norm(w)
    out = orc.kcache_update(kc, w, 1.3)
    np.testing.assert_allclose(out, kc @ dense.transition(w, 1.3).T, atol=1e-13)


# --------------------------------------------------------------------------- API consistency
def test_rows_subset_matches_full():
    rng = np.random.default_rng(31)
    B, H, L, d = 2, 3, 20, 4
    q, k, v, w = (rng.standard_normal((B, H, L, d)) for _ in range(4))
    beta = rng.random((B, H, L)) * 2
    o, lse = orc.path_attn(q, k, v, w, beta)
    rows = np.array([0, 5, 19, 20 + 7, 5 * 20 + 19])
    o2, lse2 = orc.path_attn(q, k, v, w, beta, rows=rows)
    np.testing.assert_array_equal(o2, o.reshape(-1, d)[rows])
    np.testing.assert_array_equal(lse2, lse.reshape(-1)[rows])


# --------------------------------------------------------------------------- pins catch planted mistakes
def _walk_mutant(q, k, w, beta, mutation):
    """A pure-Python copy of the walk with one planted mistake, to show the pins reject it."""
    L, d = q.shape
    S = np.full((L, L), -np.inf)
    for i in range(L):
        if mutation == "descending":
            for j in range(i + 1):
                u = q[i].copy()
                for s in range(j + 1, i + 1):  # applies H_{j+1} first: product H_i ... H_{j+1}
                    u = u - beta[s] * (w[s] @ u) * w[s]
                S[i, j] = k[j] @ u
            continue
        u = q[i].copy()
        for j in range(i, -1, -1):
            S[i, j] = k[j] @ u
            b = beta[j] / 2 if mutation == "half_beta" else beta[j]
            idx = j - 1 if (mutation == "off_by_one" and j > 0) else j
            u = u - b * (w[idx] @ u) * w[idx]
    return S


@pytest.mark.parametrize("mutation", ["descending", "half_beta", "off_by_one"])
def test_pins_reject_planted_mistakes(mutation):
    g = json.load(open(os.path.join(GOLDEN, "hand_d2_L3.json")))
    q, k, w, beta = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "w", "beta"))
    exp = np.array([[np.nan if x is None else x for x in r] for r in g["logits"]])
    mask = ~np.isnan(exp)
    good = _walk_mutant(q, k, w, beta, None)
    np.testing.assert_allclose(good[mask], exp[mask], atol=1e-12)
    bad = _walk_mutant(q, k, w, beta, mutation)
    assert np.max(np.abs(bad[mask] - exp[mask])) > 0.1


# --------------------------------------------------------------------------- relative-position bias
def _ggd_table(L, mu, alpha, p):
    """GGD-BAM prior ("Mecanismo de Atenção Bayesiana (BAM)", §"Solução Proposta: GGD-BAM"):
    b_ij = -|(j - i - mu) / alpha|^p, tabulated by the distance i - j."""
    delta = np.arange(L, dtype=np.float64)
    return -np.abs((-delta - mu) / alpha) ** p


def test_relbias_with_beta_zero_is_textbook_biased_attention():
    """beta = 0 (every transition the identity): PaTH + relative bias is softmax attention with
    the explicit bias matrix b[i, j] = rel[i - j]; reference: torch SDPA in fp64."""
    import torch
    rng = np.random.default_rng(81)
    L, d = 48, 8
    q, k, v, w, _ = _rand_case(rng, L, d)
    rel = _ggd_table(L, 0.5, 6.0, 0.7)
    o, lse = orc.path_attn(q, k, v, w, np.zeros(L), scale=0.35, rel_bias=rel)
    idx = np.arange(L)
    bias = np.where(idx[:, None] >= idx[None, :], rel[np.clip(idx[:, None] - idx[None, :], 0, L - 1)], -np.inf)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=torch.from_numpy(bias)[None], scale=0.35)[0].numpy()
    np.testing.assert_allclose(o, ref, atol=1e-12)


@pytest.mark.parametrize("seed,p", [(82, 0.6), (83, 1.3)])
def test_relbias_equals_dense_product_with_bias(seed, p):
    """Random beta: the walk oracle with a relative bias equals the explicit d x d products plus the
    bias matrix (brute force)."""
    rng = np.random.default_rng(seed)
    L, d = 20, 5
    q, k, v, w, beta = _rand_case(rng, L, d)
    rel = _ggd_table(L, 0.0, 3.0, p)
    o, lse = orc.path_attn(q, k, v, w, beta, scale=0.5, rel_bias=rel)
    o_ref, lse_ref = dense.attention(q, k, v, w, beta, scale=0.5, rel_bias=rel)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)
    # a table shifted by one position is a different operator: the pin discriminates
    o_bad, _ = orc.path_attn(q, k, v, w, beta, scale=0.5, rel_bias=np.roll(rel, 1))
    assert np.abs(o_bad - o_ref).max() > 1e-6


def test_linear_relbias_equals_constant_forget_gates():
    """ALiBi: rel[delta] = -slope * delta is the FoX bias with log f_s = -slope for every s."""
    rng = np.random.default_rng(84)
    L, d = 64, 8
    q, k, v, w, beta = _rand_case(rng, L, d)
    slope = 0.3
    o1, l1 = orc.path_attn(q, k, v, w, beta, scale=0.4, rel_bias=-slope * np.arange(L, dtype=np.float64))
    o2, l2 = orc.path_attn(q, k, v, w, beta, scale=0.4, log_f=np.full(L, -slope))
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


# --------------------------------------------------------------------------- gradients
_GRAD_NAMES = ("dq", "dk", "dv", "dw", "dbeta")


def _fd_grads(q, k, v, w, beta, dO, log_f, scale, eps=1e-6):
    """Central finite differences of sum(o * dO) through the forward oracle (brute force)."""
    args = {"q": q, "k": k, "v": v, "w": w, "beta": beta}
    if log_f is not None:
        args["log_f"] = log_f

    def loss(a):
        o, _ = orc.path_attn(a["q"], a["k"], a["v"], a["w"], a["beta"], log_f=a.get("log_f"), scale=scale)
        return float((o * dO).sum())

    out = {}
    for n, x in args.items():
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            a = dict(args)
            xp = x.copy()
            xp[idx] += eps
            a[n] = xp
            lp = loss(a)
            xm = x.copy()
            xm[idx] -= eps
            a[n] = xm
            g[idx] = (lp - loss(a)) / (2 * eps)
        out["d" + n] = g
    return out


@pytest.mark.parametrize("fox", [False, True])
@pytest.mark.parametrize("L,d,seed", [(7, 3, 91), (12, 4, 92)])
def test_bwd_matches_finite_differences(L, d, seed, fox):
    """Every gradient of the backward oracle equals central differences of the forward oracle
    (beta = 0 and beta = 2 positions included)."""
    rng = np.random.default_rng(seed)
    q, k, v, w, beta = _rand_case(rng, L, d)
    dO = rng.standard_normal((L, d))
    lf = np.log(1.0 / (1.0 + np.exp(-(3.0 + rng.standard_normal(L))))) if fox else None
    g = orc.path_attn_bwd(q, k, v, w, beta, dO, log_f=lf, scale=0.6)
    fd = _fd_grads(q, k, v, w, beta, dO, lf, 0.6)
    for n in _GRAD_NAMES + (("dlog_f",) if fox else ()):
        np.testing.assert_allclose(g[n], fd[n], rtol=0, atol=2e-8, err_msg=n)


def _torch_dense_loss(q, k, v, w, beta, dO, scale, log_f=None):
    """sum(o * dO) with every path product built from explicit d x d matrices (torch fp64)."""
    L, d = q.shape
    eye = torch.eye(d, dtype=torch.float64)
    H = [eye - beta[s] * torch.outer(w[s], w[s]) for s in range(L)]
    rows = []
    for i in range(L):
        P = eye
        logits = [None] * (i + 1)
        for j in range(i, -1, -1):  # P = H_{j+1} ... H_i, ascending
            s = scale * (k[j] @ P @ q[i])
            if log_f is not None:
                s = s + log_f[j + 1:i + 1].sum()
            logits[j] = s
            P = H[j] @ P
        rows.append(torch.softmax(torch.stack(logits), 0) @ v[: i + 1])
    return (torch.stack(rows) * dO).sum()


@pytest.mark.parametrize("fox", [False, True])
def test_bwd_matches_autograd_of_dense_products(fox):
    """Brute force: torch autograd (fp64) of the explicit-matrix PaTH forward."""
    rng = np.random.default_rng(93)
    L, d = 10, 4
    q, k, v, w, beta = _rand_case(rng, L, d)
    dO = rng.standard_normal((L, d))
    lf = -rng.uniform(0.0, 0.7, L) if fox else None
    ts = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v, w, beta)]
    tl = torch.tensor(lf, dtype=torch.float64, requires_grad=True) if fox else None
    loss = _torch_dense_loss(*ts, torch.from_numpy(dO), 0.45, tl)
    loss.backward()
    g = orc.path_attn_bwd(q, k, v, w, beta, dO, log_f=lf, scale=0.45)
    for n, t in zip(_GRAD_NAMES, ts):
        np.testing.assert_allclose(g[n], t.grad.numpy(), rtol=0, atol=1e-12, err_msg=n)
    if fox:
        np.testing.assert_allclose(g["dlog_f"], tl.grad.numpy(), rtol=0, atol=1e-12)


def test_bwd_beta_zero_is_library_attention_backward():
    """beta = 0: dq, dk, dv are those of causal softmax attention (torch SDPA autograd, fp64),
    dw vanishes and dbeta_s = -sum over (i, j<s<=i) of the transition's first-order effect."""
    rng = np.random.default_rng(94)
    L, d = 33, 8
    q, k, v, w, _ = _rand_case(rng, L, d)
    dO = rng.standard_normal((L, d))
    g = orc.path_attn_bwd(q, k, v, w, np.zeros(L), dO, scale=0.3)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], is_causal=True, scale=0.3)[0]
    (o * torch.from_numpy(dO)).sum().backward()
    for n, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        np.testing.assert_allclose(g[n], t.grad.numpy(), rtol=0, atol=1e-12, err_msg=n)
    assert np.all(g["dw"] == 0.0)
    # first order in beta_s: s_ij gains -beta_s scale (k_j.w_s)(w_s.q_i) for j < s <= i
    S = 0.3 * q @ k.T
    S = np.where(np.tril(np.ones((L, L))) > 0, S, -np.inf)
    P = np.exp(S - S.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    dS = P * (dO @ v.T - (dO * (P @ v)).sum(1, keepdims=True))
    kw, qw = k @ w.T, q @ w.T  # kw[j, s] = k_j.w_s, qw[i, s] = q_i.w_s
    exp_db = np.array([-0.3 * sum(dS[i, j] * kw[j, s] * qw[i, s] for i in range(s, L) for j in range(s))
                       for s in range(L)])
    np.testing.assert_allclose(g["dbeta"], exp_db, rtol=0, atol=1e-12)


def test_bwd_invariants():
    """Softmax rows sum to one, so sum_j dv_j = sum_i dO_i; position 0's transition acts on
    nothing, so dbeta_0 = 0, dw_0 = 0 and dlog f_0 = 0."""
    rng = np.random.default_rng(95)
    L, d = 40, 6
    q, k, v, w, beta = _rand_case(rng, L, d)
    dO = rng.standard_normal((L, d))
    g = orc.path_attn_bwd(q, k, v, w, beta, dO, log_f=-rng.uniform(0, 1, L), scale=0.5)
    np.testing.assert_allclose(g["dv"].sum(0), dO.sum(0), rtol=0, atol=1e-12)
    assert g["dbeta"][0] == 0.0 and np.all(g["dw"][0] == 0.0) and g["dlog_f"][0] == 0.0
    # batched heads give the same gradients as one head at a time
    qb, kb, vb, wb, bb = (np.stack([x, x[::-1].copy()]) for x in (q, k, v, w, beta))
    dOb = np.stack([dO, dO[::-1].copy()])
    gb = orc.path_attn_bwd(qb, kb, vb, wb, bb, dOb, scale=0.5)
    g1 = orc.path_attn_bwd(q[::-1].copy(), k[::-1].copy(), v[::-1].copy(), w[::-1].copy(), beta[::-1].copy(),
                           dO[::-1].copy(), scale=0.5)
    for n in _GRAD_NAMES:  # rows are summed by threads in parallel: equal up to rounding order
        np.testing.assert_allclose(gb[n][1], g1[n], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- gradient pins catch planted mistakes
def _bwd_walk_mutant(q, k, v, w, beta, dO, scale, mutation):
    """A pure-Python copy of the backward oracle's row walk (no forget gates) with one planted mistake,
    to show that the finite-difference pin rejects it.  Row i walks u_j = H_{j+1} ... H_i q_i down to
    j = 0, then back up with g = dloss/du: g <- H_j g + scale ds_ij k_j, the transition H_j receiving
    the outer product g u_j^T."""
    L, d = q.shape
    o, lse = orc.path_attn(q, k, v, w, beta, scale=scale)
    Delta = (dO * o).sum(1)
    grads = {n: np.zeros_like(x) for n, x in (("dq", q), ("dk", k), ("dv", v), ("dw", w), ("dbeta", beta))}
    for i in range(L):
        us, s, u = {}, {}, q[i].copy()
        for j in range(i, -1, -1):
            us[j], s[j] = u.copy(), scale * (k[j] @ u)
            u = u - beta[j] * (w[j] @ u) * w[j]
        g = np.zeros(d)
        for j in range(i + 1):
            p = np.exp(s[j] - lse[i])
            ds = p * (dO[i] @ v[j] - (0.0 if mutation == "no_delta" else Delta[i]))
            grads["dv"][j] += p * dO[i]
            grads["dk"][j] += scale * ds * us[j]
            wu, wg = w[j] @ us[j], w[j] @ g
            grads["dbeta"][j] += (wg * wu) if mutation == "dbeta_sign" else -(wg * wu)
            grads["dw"][j] += -beta[j] * (wu * g + (0.0 if mutation == "dw_one_term" else wg * us[j]))
            if mutation == "walk_order":  # the logit's share taken before the transition instead of after
                g = g + scale * ds * k[j]
                g = g - beta[j] * (w[j] @ g) * w[j]
            else:
                g = g - beta[j] * wg * w[j] + scale * ds * k[j]
        grads["dq"][i] += g
    return grads


@pytest.mark.parametrize("mutation", ["no_delta", "dbeta_sign", "dw_one_term", "walk_order"])
def test_bwd_pins_reject_planted_mistakes(mutation):
    rng = np.random.default_rng(96)
    L, d = 6, 3
    q, k, v, w, beta = _rand_case(rng, L, d)
    dO = rng.standard_normal((L, d))
    fd = _fd_grads(q, k, v, w, beta, dO, None, 0.6)
    good = _bwd_walk_mutant(q, k, v, w, beta, dO, 0.6, None)
    for n in _GRAD_NAMES:
        np.testing.assert_allclose(good[n], fd[n], rtol=0, atol=2e-8, err_msg=n)
    bad = _bwd_walk_mutant(q, k, v, w, beta, dO, 0.6, mutation)
    assert max(float(np.abs(bad[n] - fd[n]).max()) for n in _GRAD_NAMES) > 1e-3
