"""Prefill -> decode hand-off (GPU): path_prefill_kcache against the fp64 oracle.

The oracle's token-by-token decode from an empty cache (in-place key updates, "Resumo
Técnico: Atenção PaTH" §3 "Inferência") leaves exactly the transported cache
H_{L-1} ... H_{j+1} k_j; the GPU writes it from the chunked UT representation."""
import numpy as np
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import check, to_np
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _oracle_cache(x, b, h):
    f = inputs.f64
    L, d = x.k.shape[2], x.k.shape[3]
    z = np.zeros((L, d))
    _, _, kc, _ = orc.path_decode(np.zeros((0, d)), np.zeros((0, d)), z, f(x.k[b, h]), z, f(x.w[b, h]),
                                  f(x.beta[b, h]), 1.0)
    return kc


def _check_cache(got, ref, dtype, what):
    err = np.abs(got - ref)
    if dtype == "f32":
        assert err.max() <= 1e-4, (what, err.max())
    else:
        # khat and the key-side factors are bf16 and the cache is stored in bf16: a few bf16
        # roundings of values of this row's size
        bound = 2.0 ** -6 * np.abs(ref).max(axis=1, keepdims=True) + 1e-3
        assert np.all(err <= bound), (what, float((err - bound).max()))
        assert err.mean() <= 2e-3, (what, err.mean())


@pytest.mark.parametrize("dtype,B,H,L,d", [("f32", 1, 2, 200, 64), ("f32", 1, 1, 37, 16), ("bf16", 1, 2, 300, 128),
                                           ("bf16", 2, 2, 257, 64), ("bf16", 1, 1, 1, 128), ("bf16", 1, 1, 128, 128),
                                           ("bf16", 1, 2, 129, 128), ("bf16", 2, 1, 256, 128),
                                           ("bf16", 1, 1, 1500, 128)])
def test_prefill_kcache_vs_oracle(dtype, B, H, L, d):
    x = inputs.make_fwd(B, H, L, d, dtype, seed=51, edge_frac=0.05)
    ws = P.alloc_workspace(P.path_prefill_workspace_bytes(B, H, L, d, x.k.dtype), "cuda")
    kc = P.path_prefill_kcache(x.k.cuda(), x.w.cuda(), x.beta.cuda(), n_max=L + 5, workspace=ws)
    torch.cuda.synchronize()
    assert P.path_get_status(ws) == P.PATH_OK
    assert torch.count_nonzero(kc[:, :, L:]) == 0  # rows beyond the prompt untouched
    for b in range(B):
        for h in range(H):
            _check_cache(to_np(kc[b, h, :L]), _oracle_cache(x, b, h), dtype, "prefill %s b%d h%d" % (dtype, b, h))


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_prefill_then_decode_continues_the_sequence(dtype, d):
    """Prefill L0 prompt tokens, then decode T more: the decode outputs equal the oracle's
    forward rows L0 .. L0+T-1 of the whole sequence."""
    B, H, L0, T = 1, 2, 260, 12
    x = inputs.make_fwd(B, H, L0 + T, d, dtype, seed=52)
    cut = lambda t: t[:, :, :L0].contiguous().cuda()
    kc = P.path_prefill_kcache(cut(x.k), cut(x.w), x.beta[:, :, :L0].contiguous().cuda(), n_max=L0 + T)
    vc = torch.zeros_like(kc)
    vc[:, :, :L0] = x.v[:, :, :L0].cuda()
    outs = []
    for t in range(L0, L0 + T):
        step = lambda a: a[:, :, t].contiguous().cuda()
        outs.append(P.path_decode_step(step(x.q), step(x.k), step(x.v), step(x.w), x.beta[:, :, t].contiguous().cuda(),
                                       kc, vc, t, scale=x.scale))
    torch.cuda.synchronize()
    o = torch.stack(outs, dim=2)
    f = inputs.f64
    ref, _ = orc.path_attn(f(x.q), f(x.k), f(x.v), f(x.w), f(x.beta), None, x.scale)
    check(to_np(o), ref[:, :, L0:], x.q.dtype, "prefill+decode %s" % dtype)


def test_prefill_kcache_760m_shape_sampled_heads():
    """B8 H12 L4096 d128 bf16 prompt: the whole cache on the GPU, two heads on the oracle."""
    x = inputs.FWD_CONFIGS["path760m_bf16"].make()
    kc = P.path_prefill_kcache(x.k.cuda(), x.w.cuda(), x.beta.cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(kc.float()).all()
    for (b, h) in [(0, 0), (7, 11)]:
        _check_cache(to_np(kc[b, h]), _oracle_cache(x, b, h), "bf16", "prefill 760m b%d h%d" % (b, h))
