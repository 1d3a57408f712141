"""The chunked reverse mode that the backward kernels implement, restated in fp64 numpy and held
against the oracle's gradients (CPU, no GPU).

The oracle (oracle.path_attn_bwd) differentiates the per-row walk of the logit definition
(PaTH summary, §2 "Mecanismo Central": s_ij = k_j^T H_{j+1} ... H_i q_i, H_s = I - beta_s w_s w_s^T,
plus c_i - c_j with the PaTH-FoX forget gates of "Extensões: PaTH-FoX").  The kernels instead split
the sequence into chunks of C positions, the blocking of §3 "Algoritmo Estilo FlashAttention":

  prep    qbar_i = H_b ... H_i q_i (walk back to the chunk start b), khat_j = H_e ... H_{j+1} k_j
          (walk forward to the chunk end e), P_m = H_b ... H_e of each chunk, Delta_i = dO_i . o_i
  chains  for query chunk n, down the key chunks m = n-1 .. 0 with U_{n,n-1} = qbar_n and
          U_{n,m-1} = U_{n,m} P_m^T:  S = scale U khat_m^T (+ c_i - c_j), dS = P o (dO v_m^T - Delta);
          then up m = 0 .. n-1:  G_{n,m} = scale dS_{n,m} khat_m + G_{n,m-1} P_m, and dqbar_n = G_{n,n-1}
  sums    per key chunk m over n > m:  dv_m += P^T dO_n, dkhat_m += scale dS^T U, dP_m += G_{n,m-1}^T U
  local   per chunk: the diagonal block and the reversed walks that built qbar, khat and P_m

This module writes those four stages out with plain loops, so a reader can compare them with
csrc/bwd.cu and csrc/bwd_tc.cu stage by stage; the tests check that they reproduce the oracle's
dq, dk, dv, dw, dbeta (and dlog f) to fp64 rounding for several chunk sizes, ragged last chunks,
beta = 0 and beta = 2 positions, with and without forget gates.  It shares no code with the
kernels and computes nothing the oracle relies on.

The kernels form prep and local in the compact form of §3 "Representação de Transformação UT"
instead of walking (form="compact" below).  For a chunk with rows W, Q, K and D = diag(beta):

  G = W W^T,  X = (I + D triu_1 G)^-1,  A = X D   (H_a ... H_b = I - W^T A W over a..b, a principal
                                                  block of A for a sub-range)
  Qm = tril(Q W^T), Km = striu(K W^T), Y = Qm A^T, Z = Km A
  qbar = Q - Y W,  khat = K - Z W,  P = I - W^T A W,  S_diag = scale (Q K^T - Y Km^T) + c_i - c_j

and local is the reverse mode of these products (compact_local); both forms are held to the
oracle with the same bound.
"""
import numpy as np
import pytest

from oracle import oracle as orc


def _H(x, w, b):
    """H x = x - b (w . x) w for a vector x (or rows of x)."""
    return x - b * (x @ w)[..., None] * w


def _ut_factors(W, beta):
    """G = W W^T, X = (I + D triu_1 G)^-1 and A = X D: H_b ... H_e = I - W^T A W for the chunk."""
    G = W @ W.T
    X = np.linalg.inv(np.eye(len(beta)) + np.diag(beta) @ np.triu(G, 1))
    return G, X, X * beta[None, :]


def compact_prep(Q, K, W, beta):
    """qbar, khat and the chunk transition of one chunk from products (no walks)."""
    _, _, A = _ut_factors(W, beta)
    Y = np.tril(Q @ W.T) @ A.T
    Z = np.triu(K @ W.T, 1) @ A
    return Q - Y @ W, K - Z @ W, np.eye(W.shape[1]) - W.T @ A @ W


def compact_local(Q, K, V, W, beta, dO, lse, Delta, c, dQb, dKh, dP, scale):
    """The reverse mode of compact_prep and of the diagonal block's logits, for one chunk; returns
    dq, dk, the diagonal part of dv, dw, dbeta and the diagonal part of dc."""
    C = len(beta)
    G, X, A = _ut_factors(W, beta)
    le, gt = np.tril(np.ones((C, C))), np.triu(np.ones((C, C)), 1)
    Qm, Km = (Q @ W.T) * le, (K @ W.T) * gt
    Y, Z = Qm @ A.T, Km @ A
    S = scale * (Q @ K.T - Y @ Km.T) + c[:, None] - c[None, :]
    Pr = np.where(le > 0, np.exp(np.where(le > 0, S, 0.0) - lse[:, None]), 0.0)
    dS = Pr * (dO @ V.T - Delta[:, None])
    dSs = scale * dS
    dZ = -dKh @ W.T
    dY = -dQb @ W.T - dSs @ Km
    dKw = (-dSs.T @ Y + dZ @ A.T) * gt
    dQw = (dY @ A) * le
    R1, R2 = W @ dP, W @ dP.T
    dA = Km.T @ dZ + dY.T @ Qm - R1 @ W.T
    dbeta = (X * dA).sum(0)                 # A = X D
    dM = -X.T @ (dA * beta[None, :]) @ X.T  # X = M^-1, M = I + D triu_1 G
    dbeta += (dM * G * gt).sum(1)
    dG = beta[:, None] * dM * gt
    dW = (-A.T @ R1 - A @ R2 - Y.T @ dQb - Z.T @ dKh + dQw.T @ Q + dKw.T @ K + (dG + dG.T) @ W)
    dQ = dQb + dSs @ K + dQw @ W
    dK = dKh + dSs.T @ Q + dKw @ W
    return dQ, dK, Pr.T @ dO, dW, dbeta, dS.sum(1) - dS.sum(0)


def chunked_bwd(q, k, v, w, beta, dO, log_f, scale, C, form="walks"):
    L, d = q.shape
    N = -(-L // C)
    span = lambda n: (n * C, min(L, n * C + C))
    o, lse = orc.path_attn(q, k, v, w, beta, log_f=log_f, scale=scale)
    Delta = (dO * o).sum(1)
    c = np.cumsum(log_f) if log_f is not None else np.zeros(L)

    # prep: qbar, khat, P_m
    qbar, khat, Pm = np.zeros((L, d)), np.zeros((L, d)), np.zeros((N, d, d))
    for n in range(N):
        b, e = span(n)
        if form == "compact":
            qbar[b:e], khat[b:e], Pm[n] = compact_prep(q[b:e], k[b:e], w[b:e], beta[b:e])
            continue
        for i in range(b, e):
            u = q[i].copy()
            for j in range(i, b - 1, -1):
                u = _H(u, w[j], beta[j])
            qbar[i] = u
        for j in range(b, e):
            x = k[j].copy()
            for t in range(j + 1, e):
                x = _H(x, w[t], beta[t])
            khat[j] = x
        M = np.eye(d)
        for t in range(b, e):  # M <- M H_t, so P_m = H_b ... H_{e-1}
            M = M - beta[t] * np.outer(M @ w[t], w[t])
        Pm[n] = M

    # chains: per query chunk, down then up the earlier key chunks
    pairs, dqbar, dc = {}, np.zeros((L, d)), np.zeros(L)
    for n in range(1, N):
        b, e = span(n)
        U, Us, dSs = qbar[b:e].copy(), {}, {}
        for m in range(n - 1, -1, -1):
            bm, em = span(m)
            S = scale * U @ khat[bm:em].T + (c[b:e, None] - c[None, bm:em])
            Pr = np.exp(S - lse[b:e, None])
            dS = Pr * (dO[b:e] @ v[bm:em].T - Delta[b:e, None])
            dc[b:e] += dS.sum(1)
            Us[m], dSs[m] = U.copy(), dS
            U = U @ Pm[m].T
        G, Gs = None, {}
        for m in range(n):
            bm, em = span(m)
            if m >= 1:
                Gs[m] = G.copy()
            G = scale * dSs[m] @ khat[bm:em] + (G @ Pm[m] if m >= 1 else 0.0)
        dqbar[b:e] = G
        for m in range(n):
            pairs[(n, m)] = (Us[m], dSs[m], Gs.get(m))

    # sums: per key chunk over the later query chunks
    dv, dkhat, dPm = np.zeros((L, d)), np.zeros((L, d)), np.zeros((N, d, d))
    for m in range(N - 1):
        bm, em = span(m)
        for n in range(m + 1, N):
            b, e = span(n)
            U, dS, G = pairs[(n, m)]
            Pr = np.exp(scale * U @ khat[bm:em].T + (c[b:e, None] - c[None, bm:em]) - lse[b:e, None])
            dv[bm:em] += Pr.T @ dO[b:e]
            dkhat[bm:em] += scale * dS.T @ U
            dc[bm:em] -= dS.sum(0)
            if m >= 1:
                dPm[m] += G.T @ U

    # local: the diagonal block and the reversed within-chunk walks
    dq, dk, dw, db = np.zeros((L, d)), np.zeros((L, d)), np.zeros((L, d)), np.zeros(L)

    def add_dH(t, g, u):  # the transition H_t took u to H_t u and received gradient g
        wu, wg = w[t] @ u, w[t] @ g
        db[t] += -wg * wu
        dw[t] += -beta[t] * (wu * g + wg * u)

    for n in range(N):
        b, e = span(n)
        if form == "compact":
            dPn = dPm[n] if 1 <= n <= N - 2 else np.zeros((d, d))
            r = compact_local(q[b:e], k[b:e], v[b:e], w[b:e], beta[b:e], dO[b:e], lse[b:e], Delta[b:e], c[b:e],
                              dqbar[b:e], dkhat[b:e], dPn, scale)
            dq[b:e], dk[b:e], dw[b:e], db[b:e] = r[0], r[1], r[3], r[4]
            dv[b:e] += r[2]
            dc[b:e] += r[5]
            continue
        for i in range(b, e):  # (a) row i: diagonal logits and the walk that built qbar_i
            us, s, u = {}, {}, q[i].copy()
            for j in range(i, b - 1, -1):
                us[j], s[j] = u.copy(), scale * k[j] @ u + c[i] - c[j]
                u = _H(u, w[j], beta[j])
            g = dqbar[i].copy()
            for j in range(b, i + 1):
                p = np.exp(s[j] - lse[i])
                ds = p * (dO[i] @ v[j] - Delta[i])
                dv[j] += p * dO[i]
                dk[j] += scale * ds * us[j]
                dc[i] += ds
                dc[j] -= ds
                add_dH(j, g, us[j])
                g = _H(g, w[j], beta[j]) + scale * ds * k[j]
            dq[i] = g
        for j in range(b, e):  # (b) key j: the walk that built khat_j
            xs, x = {}, k[j].copy()
            for t in range(j + 1, e):
                xs[t] = x.copy()
                x = _H(x, w[t], beta[t])
            gx = dkhat[j].copy()
            for t in range(e - 1, j, -1):
                add_dH(t, gx, xs[t])
                gx = _H(gx, w[t], beta[t])
            dk[j] += gx
        for t in range(b, e):  # (c) P_n = A_t H_t B_t: dH_t = A_t^T dP_n B_t^T
            wh = w[t].copy()  # B_t^T w_t = H_{e-1} ... H_{t+1} w_t
            for s_ in range(t + 1, e):
                wh = _H(wh, w[s_], beta[s_])
            wb = w[t].copy()  # A_t w_t = H_b ... H_{t-1} w_t
            for s_ in range(t - 1, b - 1, -1):
                wb = _H(wb, w[s_], beta[s_])
            y1, y2 = dPm[n] @ wh, dPm[n].T @ wb
            db[t] += -wb @ y1
            for s_ in range(b, t):  # A_t^T y1
                y1 = _H(y1, w[s_], beta[s_])
            for s_ in range(e - 1, t, -1):  # B_t y2
                y2 = _H(y2, w[s_], beta[s_])
            dw[t] += -beta[t] * (y1 + y2)

    out = dict(dq=dq, dk=dk, dv=dv, dw=dw, dbeta=db)
    if log_f is not None:
        out["dlog_f"] = np.cumsum(dc[::-1])[::-1]  # dlog f_s = sum_{t >= s} dc_t
    return out


@pytest.mark.parametrize("form", ["walks", "compact"])
@pytest.mark.parametrize("L,d,C,fox", [(20, 4, 6, False), (23, 5, 4, True), (64, 8, 16, True), (33, 6, 8, False),
                                       (9, 3, 16, True)])
def test_chunked_backward_matches_oracle(L, d, C, fox, form):
    """Several chunks with ragged last chunks (and one chunk larger than L); beta = 0 at position 3
    and beta = 2 at position 5 where present."""
    rng = np.random.default_rng(100 + L)
    q, k, v, dO = (rng.standard_normal((L, d)) for _ in range(4))
    w = rng.standard_normal((L, d))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = rng.uniform(0.0, 2.0, L)
    if L > 5:
        beta[3], beta[5] = 0.0, 2.0
    lf = -rng.uniform(0.0, 1.0, L) if fox else None
    ref = orc.path_attn_bwd(q, k, v, w, beta, dO, log_f=lf, scale=0.5)
    got = chunked_bwd(q, k, v, w, beta, dO, lf, 0.5, C, form)
    assert set(got) == set(ref)
    for name in ref:
        scale = max(float(np.abs(ref[name]).max()), 1e-12)
        err = float(np.abs(got[name] - ref[name]).max()) / scale
        assert err <= 1e-11, (name, err)


def test_chunked_backward_chunk_size_invariant():
    """The same inputs through chunk sizes 1, 3, 7 and L give the same gradients: the blocking is a
    regrouping of one sum, not an approximation."""
    rng = np.random.default_rng(7)
    L, d = 14, 4
    q, k, v, dO = (rng.standard_normal((L, d)) for _ in range(4))
    w = rng.standard_normal((L, d))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    beta = rng.uniform(0.0, 2.0, L)
    lf = -rng.uniform(0.0, 1.0, L)
    outs = [chunked_bwd(q, k, v, w, beta, dO, lf, 0.5, C) for C in (1, 3, 7, L)]
    for o in outs[1:]:
        for name in o:
            np.testing.assert_allclose(o[name], outs[0][name], rtol=0, atol=1e-12)
