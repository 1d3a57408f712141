"""A blockwise (chunked, UT-form) restatement of the value-transport forward, in fp64 numpy, held
against the oracle's direct walk (CPU, no GPU).

The operator ("Resumo Técnico: Por que Transformações Acumuladas Extrapolam?", §"Principais
Contribuições" 3 "Proteção do Lado de Valor", with the PaTH steps H_s = I - beta_s w_s w_s^T of
"Resumo Técnico: Atenção PaTH", §2 "Mecanismo Central") is

    o_i = sum_{j <= i} alpha_ij H_i ... H_{j+1} v_j,   alpha = softmax of the PaTH(-FoX) logits.

The library computes it with two walks per query row (csrc/fwd_vt.cu).  This module writes out the
chunked form a tensor-core kernel would take, in the blocking of the PaTH page's §3 "Algoritmo
Estilo FlashAttention" and the UT representation of §3 "Representação de Transformação UT".  In a
chunk c (positions b..e, rows W_c of w) the descending product is

    H_e ... H_b = I - W_c^T B_c W_c,   B_c = (I + D_c stril(W_c W_c^T))^-1 D_c   (lower triangular),

and the product over a contiguous sub-range (j, i] is I - W^T B' W with B' the matching principal
block of B_c (a principal block of the inverse of a triangular matrix is the inverse of the same
block of the matrix).  Then, for query chunk n and key chunk m < n, with T_{n,m} = P_{n-1} ... P_{m+1}:

    vhat_j        = H_e ... H_{j+1} v_j            = rows of V - (Zv B^T) W,  Zv[j, t] = [t > j] w_t . v_j
    Vtil_{n,m}    = Vhat_m T_{n,m}^T                (Vtil_{m+1,m} = Vhat_m, Vtil_{n+1,m} = Vtil_{n,m} P_n^T)
    O_diag        = alpha_nn V_n - tril((alpha_nn Zv_n) B_n^T) W_n
    o_n           = X - tril((X W_n^T) B_n^T) W_n + O_diag,   X = sum_{m<n} alpha_nm Vtil_{n,m}

(the last line applies H_i ... H_b row by row).  Each mask pairs one index of B with one side:
the projection index t with the key (t > j), the output index s with the query (s <= i), so both
separate into masked products, as they do for the logits' Y (-Z)^T on the key side.  Every step is
a product of chunk-sized matrices; the tests check the whole against the oracle to fp64 rounding
for several chunk sizes, ragged last chunks, beta = 0 and beta = 2 positions, with and without
forget gates.  Nothing here is used by the library or by the oracle.
"""
import numpy as np
import pytest

from oracle import oracle as orc


def _ut_lower(Wc, bc):
    """B with H_e ... H_b = I - Wc^T B Wc (rows of Wc in position order b..e)."""
    G = Wc @ Wc.T
    Dm = np.diag(bc)
    return np.linalg.solve(np.eye(len(bc)) + Dm @ np.tril(G, -1), Dm)


def chunked_vt_forward(q, k, v, w, beta, log_f, scale, C):
    L, d = q.shape
    N = -(-L // C)
    span = lambda n: (n * C, min(L, n * C + C))
    S = orc.path_logits(q, k, w, beta, log_f=log_f, scale=scale)
    alpha = np.exp(S - S.max(axis=1, keepdims=True))
    alpha /= alpha.sum(axis=1, keepdims=True)

    B, P, Vhat, Zv = [], [], [], []
    for c in range(N):
        b, e = span(c)
        Wc, Vc = w[b:e], v[b:e]
        Bc = _ut_lower(Wc, beta[b:e])
        Zc = np.triu(Vc @ Wc.T, 1)  # [j, t] = w_t . v_j for t > j
        B.append(Bc)
        P.append(np.eye(d) - Wc.T @ Bc @ Wc)
        Zv.append(Zc)
        Vhat.append(Vc - (Zc @ Bc.T) @ Wc)

    o = np.zeros((L, d))
    for n in range(N):
        b, e = span(n)
        Wn, Bn = w[b:e], B[n]
        an = alpha[b:e, b:e]
        o_diag = an @ v[b:e] - np.tril((an @ Zv[n]) @ Bn.T) @ Wn
        X = np.zeros((e - b, d))
        for m in range(n):
            bm, em = span(m)
            Vt = Vhat[m]
            for c in range(m + 1, n):  # Vtil_{c+1,m} = Vtil_{c,m} P_c^T
                Vt = Vt @ P[c].T
            X += alpha[b:e, bm:em] @ Vt
        o[b:e] = X - np.tril((X @ Wn.T) @ Bn.T) @ Wn + o_diag
    return o


def _inputs(L, d, seed, fox, edges):
    rng = np.random.default_rng(seed)
    q, k, v, w = (rng.standard_normal((L, d)) for _ in range(4))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = rng.uniform(0.0, 2.0, L)
    if edges:
        beta[rng.choice(L, 3, replace=False)] = 0.0
        beta[rng.choice(L, 3, replace=False)] = 2.0
    log_f = np.log(rng.uniform(0.6, 1.0, L)) if fox else None
    return q, k, v, w, beta, log_f


@pytest.mark.parametrize("L,d,C,fox,edges", [(13, 4, 4, False, False), (13, 4, 3, True, True), (17, 6, 5, False, True),
                                             (16, 8, 16, True, False), (9, 3, 1, False, True), (20, 5, 7, True, True)])
def test_chunked_value_transport_matches_oracle(L, d, C, fox, edges):
    q, k, v, w, beta, log_f = _inputs(L, d, seed=L * 31 + C, fox=fox, edges=edges)
    scale = d ** -0.5
    got = chunked_vt_forward(q, k, v, w, beta, log_f, scale, C)
    ref, _ = orc.path_attn(q, k, v, w, beta, log_f=log_f, scale=scale, value_transport=True)
    assert np.abs(got - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_sub_range_factor_is_the_principal_block():
    """H_i ... H_{j+1} = I - W^T B' W over positions j+1..i, with B' the principal block of the chunk's B."""
    q, k, v, w, beta, _ = _inputs(7, 5, seed=3, fox=False, edges=True)
    B = _ut_lower(w, beta)
    for i in range(7):
        for j in range(-1, i):
            M = np.eye(5)
            for s in range(i, j, -1):
                M = M @ (np.eye(5) - beta[s] * np.outer(w[s], w[s]))
            Ws, Bs = w[j + 1:i + 1], B[j + 1:i + 1, j + 1:i + 1]
            assert np.abs(M - (np.eye(5) - Ws.T @ Bs @ Ws)).max() <= 1e-13
