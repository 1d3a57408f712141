"""The allocation-free decode step against the workspace decode step (GPU).

path_decode_step_noalloc serves callers that cannot allocate device memory while
decoding (a runtime whose device memory belongs to another allocator, or a serving
loop that must not call cudaMalloc once running): it takes no workspace and uses the
library's built-in 8 MiB scratch instead.  Here it must reproduce path_decode_step bit
for bit (output, log-sum-exp and updated caches) on two calls in a row, so that the
second call also shows nothing stale from the first leaks through the shared scratch,
and at the largest size the scratch accepts.

This file is collected last on purpose: a run that stops at its first failure has
already run every other test by the time it gets here.
"""
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,B,H,n0,d", [("bf16", 2, 3, 5000, 128), ("f32", 1, 4, 2100, 64)])
def test_noalloc_decode_matches_workspace_decode_twice(dtype, B, H, n0, d):
    T = 2
    kc, vc = inputs.make_decode_cache(B, H, n0, d, n0 + T, dtype, seed=31)
    q, k, v, w, beta = (t.cuda() for t in inputs.make_decode_steps(B, H, d, T, dtype, seed=31))
    ka, va = kc.cuda(), vc.cuda()
    kb, vb = ka.clone(), va.clone()
    scale = d ** -0.5
    for t in range(T):  # two calls in a row
        oa, la = P.path_decode_step(q[t], k[t], v[t], w[t], beta[t], ka, va, n0 + t, scale=scale, lse=True)
        ob, lb = P.path_decode_step_noalloc(q[t], k[t], v[t], w[t], beta[t], kb, vb, n0 + t, scale=scale, lse=True)
        torch.cuda.synchronize()
        # the same kernels on the same grid: bit for bit
        assert torch.equal(oa, ob) and torch.equal(la, lb)
        assert torch.equal(ka, kb) and torch.equal(va, vb)


def test_noalloc_decode_at_the_largest_accepted_size():
    """B64 H12 d128 bf16 with n_max = 43008, the largest cache whose split partials fit the 8 MiB
    scratch, at its last row (n_cached = 43007): the writes reach the end of the array.  The caches
    are random device data (about 17 GB for the two copies of K and V); both entry points must
    agree bit for bit, and one row more is rejected before any launch."""
    B, H, d, n_max = 64, 12, 128, 43008
    n = n_max - 1
    g = torch.Generator(device="cuda").manual_seed(77)
    ka = torch.randn((B, H, n_max, d), generator=g, device="cuda").to(torch.bfloat16)
    va = torch.randn((B, H, n_max, d), generator=g, device="cuda").to(torch.bfloat16)
    kb, vb = ka.clone(), va.clone()
    q, k, v = (torch.randn((B, H, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    w = torch.nn.functional.normalize(torch.randn((B, H, d), generator=g, device="cuda"), dim=-1).to(torch.bfloat16)
    beta = 2 * torch.sigmoid(torch.randn((B, H), generator=g, device="cuda"))
    oa, la = P.path_decode_step(q, k, v, w, beta, ka, va, n, lse=True)
    ob, lb = P.path_decode_step_noalloc(q, k, v, w, beta, kb, vb, n, lse=True)
    torch.cuda.synchronize()
    assert torch.isfinite(oa.float()).all()
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    assert torch.equal(ka, kb) and torch.equal(va, vb)
    del ka, va, kb, vb
    kc = torch.empty((B, H, n_max + 1, d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(P.PathError) as ei:
        P.path_decode_step_noalloc(q, k, v, w, beta, kc, kc, n, lse=True)
    assert ei.value.code == P.PATH_ERR_WORKSPACE
