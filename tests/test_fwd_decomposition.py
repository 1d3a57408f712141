"""The blocked forward that the kernels implement, restated in fp64 numpy and held against the
oracle's walk (CPU, no GPU).

The oracle walks every query backwards through the transitions (PaTH summary, §2 "Mecanismo
Central").  The kernels follow §3 "Algoritmo Estilo FlashAttention" and "Representação de
Transformação UT" instead: per chunk of C rows (W, Q, K, beta of the chunk, D = diag(beta))

  A     = (I + D triu_1(W W^T))^{-1} D          the UT factor (upper triangular)
  qhat  = Q - Y W,  Y = tril(Q W^T) A^T          each query carried to its chunk's start
  khat  = K - (Z A) W,  Z = triu_1(K W^T)        each key carried to its chunk's end
  -U    = -A^T W                                 so that x P_m^T = x - (x W^T) U for a row x
  P - I = -W^T (A W)                             the chunk's transition P_m = H_b ... H_e, minus I
  S_nn  = scale (Q K^T - Y Z^T), j <= i          the diagonal block

and a query tile then walks the earlier chunks m = n-1 .. 0 with q~ <- qhat_n:
S_nm = scale q~ khat_m^T, then q~ <- q~ P_m^T, the logits of all blocks entering one softmax (with the
forget-gate bias c_i - c_j of "Extensões: PaTH-FoX" when given).  The transition is taken in one of
two equal forms: q~ + (q~ W_m^T)(-U_m) (the fp32 CUDA-core scan) or q~ + q~ (P_m - I)^T (the bf16
tensor-core scan, one d x d product).  This module
writes those steps out with dense numpy products, and the tests check that they reproduce the
oracle's o and lse to fp64 rounding for several chunk sizes, ragged last chunks and beta = 0 /
beta = 2 positions; the prefill -> decode hand-off's suffix products are checked against explicit
walks the same way.  It shares no code with the kernels and computes nothing the oracle relies on.
"""
import numpy as np
import pytest

from oracle import oracle as orc


def chunk_factors(Wc, Qc, Kc, bc):
    """The per-chunk UT quantities of one (padded) chunk."""
    C = Wc.shape[0]
    D = np.diag(bc)
    A = np.linalg.solve(np.eye(C) + D @ np.triu(Wc @ Wc.T, 1), D)
    Y = np.tril(Qc @ Wc.T) @ A.T
    Z = np.triu(Kc @ Wc.T, 1)
    return dict(A=A, Y=Y, Z=Z, qhat=Qc - Y @ Wc, khat=Kc - (Z @ A) @ Wc, negU=-A.T @ Wc, PmI=-Wc.T @ (A @ Wc))


def blocked_fwd(q, k, v, w, beta, scale, C, log_f=None, transition="two_products"):
    L, d = q.shape
    N = -(-L // C)
    Lp = N * C
    pad = lambda x: np.concatenate([x, np.zeros((Lp - L,) + x.shape[1:])])
    Q, K, V, W, B = pad(q), pad(k), pad(v), pad(w), pad(beta)
    c = pad(np.cumsum(log_f)) if log_f is not None else np.zeros(Lp)
    f = [chunk_factors(W[n * C:(n + 1) * C], Q[n * C:(n + 1) * C], K[n * C:(n + 1) * C], B[n * C:(n + 1) * C])
         for n in range(N)]
    o, lse = np.zeros((Lp, d)), np.zeros(Lp)
    for n in range(N):
        rows = slice(n * C, (n + 1) * C)
        S = np.full((C, Lp), -np.inf)
        Sd = scale * (Q[rows] @ K[rows].T - f[n]["Y"] @ f[n]["Z"].T)
        S[:, rows] = np.where(np.tril(np.ones((C, C))) > 0, Sd, -np.inf)
        qt = f[n]["qhat"].copy()
        for m in range(n - 1, -1, -1):
            cols = slice(m * C, (m + 1) * C)
            S[:, cols] = scale * qt @ f[m]["khat"].T
            if transition == "two_products":
                qt = qt + (qt @ W[cols].T) @ f[m]["negU"]
            else:
                qt = qt + qt @ f[m]["PmI"].T
        S = S + (c[rows, None] - c[None, :])
        S[:, L:] = -np.inf  # padded keys
        mx = S.max(1, keepdims=True)
        p = np.exp(S - mx)
        o[rows] = (p @ V) / p.sum(1, keepdims=True)
        lse[rows] = mx[:, 0] + np.log(p.sum(1))
    return o[:L], lse[:L]


def _case(rng, L, d):
    q, k, v = (rng.standard_normal((L, d)) for _ in range(3))
    w = rng.standard_normal((L, d))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = 2.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    if L > 6:
        beta[2], beta[6] = 0.0, 2.0
    return q, k, v, w, beta


@pytest.mark.parametrize("transition", ["two_products", "pm"])
@pytest.mark.parametrize("L,d,C,fox", [(1, 4, 4, False), (13, 4, 4, False), (30, 6, 8, True), (64, 16, 16, False),
                                       (77, 8, 32, True), (40, 8, 64, False)])
def test_blocked_forward_matches_oracle(L, d, C, fox, transition):
    rng = np.random.default_rng(200 + L)
    q, k, v, w, beta = _case(rng, L, d)
    lf = -rng.uniform(0.0, 1.0, L) if fox else None
    o_ref, lse_ref = orc.path_attn(q, k, v, w, beta, log_f=lf, scale=0.5)
    o, lse = blocked_fwd(q, k, v, w, beta, 0.5, C, log_f=lf, transition=transition)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-11)


def test_chunk_transition_is_the_ordered_product():
    """P_m - I from the UT factor equals H_b H_(b+1) ... H_e - I, built as explicit d x d matrices in
    ascending order (beta = 0 and beta = 2 positions included); the descending product differs."""
    rng = np.random.default_rng(17)
    C, d = 10, 6
    q, k, _, w, beta = _case(rng, C, d)
    f = chunk_factors(w, q, k, beta)
    P = np.eye(d)
    for t in range(C):
        P = P @ (np.eye(d) - beta[t] * np.outer(w[t], w[t]))
    np.testing.assert_allclose(f["PmI"], P - np.eye(d), rtol=0, atol=1e-12)
    Pdesc = np.eye(d)
    for t in range(C - 1, -1, -1):
        Pdesc = Pdesc @ (np.eye(d) - beta[t] * np.outer(w[t], w[t]))
    assert np.abs(Pdesc - P).max() > 1e-3


def test_chunk_factors_carry_rows_to_the_chunk_ends():
    """qhat_i = H_b ... H_i q_i and khat_j = H_e ... H_{j+1} k_j, by explicit walks."""
    rng = np.random.default_rng(9)
    C, d = 12, 5
    q, k, _, w, beta = _case(rng, C, d)
    f = chunk_factors(w, q, k, beta)
    H = lambda x, t: x - beta[t] * (w[t] @ x) * w[t]
    for i in range(C):
        u = q[i].copy()
        for t in range(i, -1, -1):
            u = H(u, t)
        np.testing.assert_allclose(f["qhat"][i], u, rtol=0, atol=1e-12)
        x = k[i].copy()
        for t in range(i + 1, C):
            x = H(x, t)
        np.testing.assert_allclose(f["khat"][i], x, rtol=0, atol=1e-12)


def test_blocked_prefill_cache_matches_walks():
    """The prefill -> decode hand-off (§3 "Inferência"): the cache a prompt of L tokens leaves is
    k~_j = H_{L-1} ... H_{j+1} k_j.  Blocked as the hand-off kernels do it: khat_j to its chunk's end,
    then k~_j^T = khat_j^T N_{m+1} with the suffix products N_c = P_c ... P_last built right to left as
    N_c = N_{c+1} - W_c^T (V_c N_{c+1}), V_c = A_c W_c (so P_c = I - W_c^T V_c)."""
    rng = np.random.default_rng(31)
    L, d, C = 45, 6, 8
    q, k, _, w, beta = _case(rng, L, d)
    N = -(-L // C)
    Lp = N * C
    pad = lambda x: np.concatenate([x, np.zeros((Lp - L,) + x.shape[1:])])
    Q, K, W, B = pad(q), pad(k), pad(w), pad(beta)
    f = [chunk_factors(W[n * C:(n + 1) * C], Q[n * C:(n + 1) * C], K[n * C:(n + 1) * C], B[n * C:(n + 1) * C])
         for n in range(N)]
    cache = np.zeros((Lp, d))
    Nsuf = np.eye(d)  # N_{c+1}, empty past the last chunk
    for c in range(N - 1, -1, -1):
        cache[c * C:(c + 1) * C] = f[c]["khat"] @ Nsuf
        Wc = W[c * C:(c + 1) * C]
        Nsuf = Nsuf - Wc.T @ ((f[c]["A"] @ Wc) @ Nsuf)
    for j in range(L):
        x = k[j].copy()
        for t in range(j + 1, L):
            x = x - beta[t] * (w[t] @ x) * w[t]
        np.testing.assert_allclose(cache[j], x, rtol=0, atol=1e-12)


def test_blocked_ut_factor_by_doubling_merges():
    """The UT prep's blocked A = (I + D triu_1(G))^{-1} D: 16 x 16 diagonal blocks of X by back
    substitution scaled by D, then doubling merges A_PQ = -A_PP G_PQ A_QQ at block sizes 16, 32, 64
    (which is X_PQ D_Q for X_PQ = -X_PP D_P G_PQ X_QQ) equal the direct solve, with beta = 0 and
    beta = 2 positions."""
    rng = np.random.default_rng(23)
    C, d = 128, 32
    w = rng.standard_normal((C, d))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = 2.0 / (1.0 + np.exp(-rng.standard_normal(C)))
    beta[[3, 40, 77]] = 0.0
    beta[[5, 64, 100]] = 2.0
    G = w @ w.T
    D = np.diag(beta)
    A_ref = np.linalg.solve(np.eye(C) + D @ np.triu(G, 1), D)
    A = np.zeros((C, C))
    for b in range(0, C, 16):
        blk = slice(b, b + 16)
        X = np.linalg.inv(np.eye(16) + np.diag(beta[blk]) @ np.triu(G[blk, blk], 1))
        A[blk, blk] = X @ np.diag(beta[blk])
    for S in (16, 32, 64):
        for P0 in range(0, C, 2 * S):
            P, Q = slice(P0, P0 + S), slice(P0 + S, P0 + 2 * S)
            A[P, Q] = -A[P, P] @ G[P, Q] @ A[Q, Q]
    np.testing.assert_allclose(A, A_ref, rtol=0, atol=1e-12)
