"""The hi + lo bf16 operand split that the tensor-core kernels use for quantities that are not exact
in bf16 (the UT factor A, tril(Q W^T), Y, Z, Z A, the transported-query master q~, the backward's
carried U and G, the chunk transitions P_m), checked on the CPU against its error bound.

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
