"""Brute-force second oracle: explicit d x d transition matrices — TEST INFRASTRUCTURE.

Builds every H_s = I - beta_s w_s w_s^T of "Resumo Técnico: Atenção PaTH"
(gist.science/pt/paper/2505.16381), §2 "Mecanismo Central", as a dense numpy
fp64 matrix and multiplies the path product prod_{s=j+1}^{i} H_s out in full
(ascending order, H_{j+1} on the left), then takes the logit
k_j^T (prod) q_i of the attention-logit equation.  Cost is O(L^2 d^3): tiny
inputs only.  Shares nothing with oracle/path_oracle.c beyond the definition.
"""
from __future__ import annotations

import numpy as np


def transition(w_s, beta_s):
    """H_s = I - beta_s w_s w_s^T as a dense d x d matrix."""
    w_s = np.asarray(w_s, dtype=np.float64)
    return np.eye(w_s.shape[0]) - float(beta_s) * np.outer(w_s, w_s)


def path_product(w, beta, j, i):
    """prod_{s=j+1}^{i} H_s, multiplied left to right (H_{j+1} first); I when j >= i."""
    d = w.shape[1]
    P = np.eye(d)
    for s in range(j + 1, i + 1):
        P = P @ transition(w[s], beta[s])
    return P


def logits(q, k, w, beta, scale=1.0, log_f=None, rel_bias=None):
    """[L, L] PaTH logits of one head; -inf above the diagonal.  rel_bias[i - j] (optional)
    is added unscaled to entry (i, j)."""
    q, k, w, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, w, beta))
    L = q.shape[0]
    S = np.full((L, L), -np.inf)
    for i in range(L):
        for j in range(i + 1):
            s = scale * (k[j] @ path_product(w, beta, j, i) @ q[i])
            if log_f is not None:
                s += sum(float(log_f[t]) for t in range(j + 1, i + 1))
            if rel_bias is not None:
                s += float(rel_bias[i - j])
            S[i, j] = s
    return S


def attention(q, k, v, w, beta, scale=1.0, log_f=None, rel_bias=None):
    """Causal softmax attention over the dense-product logits; returns (o [L, d], lse [L])."""
    S = logits(q, k, w, beta, scale, log_f, rel_bias)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    o = (P / l) @ np.asarray(v, dtype=np.float64)
    return o, (m + np.log(l))[:, 0]
