"""Seeded input generators: determinism and the stated distributions (CPU only)."""
import torch

from attention_causal_attn_fwd_gb300 import inputs


def test_fwd_inputs_deterministic_and_shaped():
    a = inputs.FWD_CONFIGS["tiny_f32"].make()
    b = inputs.FWD_CONFIGS["tiny_f32"].make()
    for x, y in zip((a.q, a.k, a.v, a.w, a.beta), (b.q, b.k, b.v, b.w, b.beta)):
        assert torch.equal(x, y)
    assert a.q.shape == (1, 1, 64, 16) and a.q.dtype == torch.float32
    assert torch.allclose(a.w.norm(dim=-1), torch.ones(1, 1, 64), atol=1e-6)
    assert float(a.beta.min()) > 0 and float(a.beta.max()) < 2
    assert a.scale == 0.25


def test_small_config_edge_fractions():
    x = inputs.FWD_CONFIGS["small_bf16"].make()
    n = x.beta.numel()
    f0 = float((x.beta == 0).sum()) / n
    f2 = float((x.beta == 2).sum()) / n
    assert 0.04 < f0 < 0.06 and 0.04 < f2 < 0.06
    assert x.q.dtype == torch.bfloat16 and x.beta.dtype == torch.float32


def test_fox_gates_are_log_sigmoid():
    x = inputs.make_fwd(1, 2, 256, 16, "bf16", 3, fox=True)
    assert x.log_f is not None and float(x.log_f.max()) < 0
    assert abs(float(x.log_f.mean()) - (-0.07)) < 0.05  # E[log sigmoid(N(3,1))] ~ -0.07


def test_decode_cache_heads_regenerate_alone():
    kc, vc = inputs.make_decode_cache(2, 3, 40, 8, 48, "bf16", seed=4)
    ks, vs = inputs.make_decode_cache(2, 3, 40, 8, 48, "bf16", seed=4, heads=[4, 1])
    assert torch.equal(ks[0], kc.view(6, 48, 8)[4, :40])
    assert torch.equal(vs[1], vc.view(6, 48, 8)[1, :40])
    assert torch.count_nonzero(kc[:, :, 40:]) == 0
