"""The hi + lo bf16 operand split that the tensor-core kernels use for quantities that are not exact
in bf16 (the UT factor A and its doubling merge, tril(Q W^T), Y, Z, A W, the backward's carried U
and G, the chunk transitions P_m), checked on the CPU against its error bound.

x = hi + lo + r with hi = bf16(x), lo = bf16(x - hi): |x - hi| <= 2^-9 |x| and |r| <= 2^-18 |x|
(round to nearest, 8 significant bits).  A product a b is taken as hi_a hi_b + hi_a lo_b + lo_a hi_b,
each term exact in fp32, so it misses lo_a lo_b and the r terms: at most 3 * 2^-18 |a| |b| + O(2^-27).
Summed over K terms with fp32 accumulation (one rounding of 2^-24 per add) the error of each output
stays below (3 * 2^-18 + K * 2^-24) * sum_k |a_ik| |b_kj|, against 2^-8 for bf16 operands alone.
"""
import numpy as np
import pytest
import torch


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def _split(x):
    hi = _bf16(x)
    return hi, _bf16(x.astype(np.float32) - hi)


@pytest.mark.parametrize("M,K,N,seed", [(128, 128, 128, 0), (128, 64, 128, 1), (64, 128, 32, 2)])
def test_hi_lo_split_product_bound(M, K, N, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)).astype(np.float32) * np.exp(rng.uniform(-3, 3, (M, 1))).astype(np.float32)
    b = rng.standard_normal((K, N)).astype(np.float32)
    exact = a.astype(np.float64) @ b.astype(np.float64)
    ha, la = _split(a)
    hb, lb = _split(b)
    # three MMAs with fp32 accumulation; each elementwise product of two bf16 values is exact in fp32
    split = (ha @ hb + ha @ lb + la @ hb).astype(np.float64)
    mag = np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64)
    bound = (3 * 2.0 ** -18 + 3 * K * 2.0 ** -24) * mag
    assert np.all(np.abs(split - exact) <= bound)
    # bf16 operands alone are three orders of magnitude worse, which is why the split is used
    plain = (ha @ hb).astype(np.float64)
    assert np.max(np.abs(plain - exact) / mag) > 50 * np.max(np.abs(split - exact) / mag)


def test_bf16_unit_w_transitions_stay_within_the_fox_skip_margin():
    """The PaTH-FoX far-block skip bounds a transported logit by 2 |q| max |khat|: each H_s is
    non-expansive for beta in [0, 2] and unit w, and the factor 2 is the margin for w rounded to bf16,
    whose squared norm is off by at most ~2^-8 so that one transition can stretch the component
    along w by at most 1 + 2^-7.  For random bf16 unit w (the inputs' recipe) the growth of a vector
    walked through 4096 transitions with beta = 2 (the expanding extreme) stays far inside 2."""
    rng = np.random.default_rng(41)
    L, d = 4096, 128
    w = rng.standard_normal((L, d)).astype(np.float32)
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    w = _bf16(w).astype(np.float64)
    n2 = (w * w).sum(1)
    assert np.max(np.abs(n2 - 1.0)) <= 2.0 ** -8
    for trial in range(4):
        x = rng.standard_normal(d)
        x0 = np.linalg.norm(x)
        peak = 1.0
        for s in range(L):
            x = x - 2.0 * (w[s] @ x) * w[s]
            peak = max(peak, np.linalg.norm(x) / x0)
        assert peak < 1.05, peak


def test_hi_lo_merge_at_64_keeps_the_solve_accurate():
    """The UT prep's last doubling merge, A_PQ = -A_PP (G_PQ A_QQ), runs as two hi/lo products on the
    tensor cores (the intermediate T = G_PQ A_QQ rounded to fp32 and split again).  With unit w and
    beta in [0, 2] (5 % each at 0 and 2) the merged block stays within 1e-4 of max |A_PQ| of the exact
    solve, the precision its own hi/lo operands carry into the later products (2^-16 relative)."""
    rng = np.random.default_rng(11)
    C, d = 128, 128
    worst = 0.0
    for _ in range(8):
        w = rng.standard_normal((C, d))
        w /= np.linalg.norm(w, axis=1, keepdims=True)
        w = _bf16(w).astype(np.float64)
        beta = 2.0 / (1.0 + np.exp(-2.0 * rng.standard_normal(C)))
        u = rng.random(C)
        beta[u < 0.05] = 0.0
        beta[(u >= 0.05) & (u < 0.10)] = 2.0
        G = (w @ w.T).astype(np.float32).astype(np.float64)
        A = np.linalg.solve(np.eye(C) + np.diag(beta) @ np.triu(G, 1), np.diag(beta))
        P, Q = slice(0, 64), slice(64, 128)
        gh, gl = _split(G[P, Q])
        ah, al = _split(A[Q, Q])
        T = (gh @ ah + gh @ al + gl @ ah).astype(np.float32)
        th, tl = _split(T)
        ph, pl = _split(A[P, P])
        apq = -(ph.astype(np.float64) @ th + ph.astype(np.float64) @ tl + pl.astype(np.float64) @ th)
        worst = max(worst, np.abs(apq - A[P, Q]).max() / np.abs(A[P, Q]).max())
    assert worst <= 1e-4, worst
