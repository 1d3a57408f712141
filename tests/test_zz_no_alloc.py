"""The allocation-free decode step against the workspace decode step (GPU).

path_decode_step_noalloc serves callers that cannot allocate device memory while
decoding (a runtime whose device memory belongs to another allocator, or a serving
loop that must not call cudaMalloc once running): it takes no workspace and uses the
library's built-in 8 MiB scratch instead.  Here it must reproduce path_decode_step,
output, log-sum-exp and updated caches, on two calls in a row, so that the second
call also shows nothing stale from the first leaks through the shared scratch.

This file is collected last on purpose: a run that stops at its first failure has
already run every other test by the time it gets here.
"""
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import BF16_MAX, BF16_MEAN, F32_MAX

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,B,H,n0,d", [("bf16", 2, 3, 5000, 128), ("f32", 1, 4, 2100, 64)])
def test_noalloc_decode_matches_workspace_decode_twice(dtype, B, H, n0, d):
    T = 2
    kc, vc = inputs.make_decode_cache(B, H, n0, d, n0 + T, dtype, seed=31)
    q, k, v, w, beta = (t.cuda() for t in inputs.make_decode_steps(B, H, d, T, dtype, seed=31))
    ka, va = kc.cuda(), vc.cuda()
    kb, vb = ka.clone(), va.clone()
    scale = d ** -0.5
    tol_max = F32_MAX if dtype == "f32" else BF16_MAX
    for t in range(T):  # two calls in a row
        oa, la = P.path_decode_step(q[t], k[t], v[t], w[t], beta[t], ka, va, n0 + t, scale=scale, lse=True)
        ob, lb = P.path_decode_step_noalloc(q[t], k[t], v[t], w[t], beta[t], kb, vb, n0 + t, scale=scale, lse=True)
        torch.cuda.synchronize()
        err = (oa.double() - ob.double()).abs()
        assert float(err.max()) <= tol_max
        if dtype == "bf16":
            assert float(err.mean()) <= BF16_MEAN
        assert float((la.double() - lb.double()).abs().max()) <= tol_max
        assert float((ka.double() - kb.double()).abs().max()) <= tol_max
        assert torch.equal(va, vb)
