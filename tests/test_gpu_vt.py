"""GPU value-side transport (path_attn_fwd_vt, path_decode_step_vt, through the C ABI) against the
fp64 value-transport oracle ("Resumo Técnico: Por que Transformações Acumuladas Extrapolam?",
§"Principais Contribuições" 3: the route transport H_i ... H_{j+1} applied to the values as well as
to the keys)."""
import numpy as np
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import check, check_lse, cuda, to_np
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _vt_fwd(x):
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    B, H, L, d = x.q.shape
    ws = P.alloc_workspace(P.load().path_attn_fwd_vt_workspace_bytes(B, H, L, d, P._DT[x.q.dtype]), "cuda")
    o, lse = P.path_attn_fwd_vt(*args, log_f=cuda(x.log_f), scale=x.scale, lse=True, workspace=ws)
    torch.cuda.synchronize()
    assert P.path_get_status(ws) == P.PATH_OK
    return o, lse


@pytest.mark.parametrize("dtype,B,H,L,d,fox", [("f32", 1, 1, 64, 16, False), ("f32", 1, 2, 77, 32, True),
                                               ("bf16", 2, 4, 1024, 64, False), ("bf16", 1, 2, 300, 128, True),
                                               ("bf16", 1, 1, 1, 128, False), ("f32", 2, 1, 129, 128, False)])
def test_fwd_vt_vs_oracle(dtype, B, H, L, d, fox):
    x = inputs.make_fwd(B, H, L, d, dtype, seed=500 + L, fox=fox, edge_frac=0.05)
    o, lse = _vt_fwd(x)
    f = inputs.f64
    o_ref, lse_ref = orc.path_attn(*(f(t) for t in (x.q, x.k, x.v, x.w, x.beta)),
                                   None if x.log_f is None else f(x.log_f), x.scale, value_transport=True)
    check(to_np(o), o_ref, x.q.dtype, "fwd vt %s %s" % (dtype, (B, H, L, d)))
    check_lse(to_np(lse), lse_ref, x.q.dtype, "fwd vt lse")


def test_fwd_vt_beta_zero_equals_plain_forward():
    """With every beta = 0 the route is the identity: the value-transport forward equals path_attn_fwd."""
    x = inputs.make_fwd(1, 2, 500, 128, "bf16", seed=510)
    x.beta.zero_()
    o_vt, _ = _vt_fwd(x)
    o = P.path_attn_fwd(*(cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)), scale=x.scale)
    torch.cuda.synchronize()
    assert float((o_vt.float() - o.float()).abs().max()) <= 2e-2


@pytest.mark.parametrize("dtype,H,d,fox", [("bf16", 12, 128, True), ("f32", 16, 64, False)])
def test_fwd_vt_second_band(dtype, H, d, fox):
    """More groups of 4 query rows than warps in the launch (L = 1024: 3072 groups on 2432 warps at
    d = 128, 4096 on 3648 at d = 64), so warps take a second group, in the reversed order."""
    x = inputs.make_fwd(1, H, 1024, d, dtype, seed=530 + d, fox=fox, edge_frac=0.05)
    o, lse = _vt_fwd(x)
    f = inputs.f64
    o_ref, lse_ref = orc.path_attn(*(f(t) for t in (x.q, x.k, x.v, x.w, x.beta)),
                                   None if x.log_f is None else f(x.log_f), x.scale, value_transport=True)
    check(to_np(o), o_ref, x.q.dtype, "fwd vt second band %s d%d" % (dtype, d))
    check_lse(to_np(lse), lse_ref, x.q.dtype, "fwd vt second band lse")


def _sampled_rows(BH, L, n, seed):
    rng = np.random.default_rng(seed)
    heads = np.arange(BH)
    fixed = np.concatenate([heads * L, heads * L + L - 1, heads * L + L - 2])
    return np.unique(np.concatenate([fixed, rng.integers(0, BH * L, n)]))


@pytest.mark.parametrize("B,H,L,d,fox", [(8, 12, 4096, 128, False), (1, 12, 4096, 128, True),
                                         (2, 2, 9000, 128, True), (1, 2, 9000, 64, True)])
def test_fwd_vt_long_sampled_rows(B, H, L, d, fox):
    """The timed value-transport workload (B8 H12 L4096 d128 bf16), its PaTH-FoX variant at B1, and
    PaTH-FoX sequences longer than 8192 tokens (blockwise at d = 128, row walks at d = 64), checked
    on sampled rows: the first and last two of every head and 64 drawn at random."""
    x = inputs.make_fwd(B, H, L, d, "bf16", seed=540 + L, fox=fox)
    o, lse = _vt_fwd(x)
    rows = _sampled_rows(B * H, L, 64, seed=L)
    f = inputs.f64
    o_ref, lse_ref = orc.path_attn(*(f(t) for t in (x.q, x.k, x.v, x.w, x.beta)),
                                   None if x.log_f is None else f(x.log_f), x.scale, rows=rows,
                                   value_transport=True)
    check(to_np(o).reshape(-1, d)[rows], o_ref, x.q.dtype, "fwd vt sampled L%d" % L)
    check_lse(to_np(lse).reshape(-1)[rows], lse_ref, x.q.dtype, "fwd vt sampled lse L%d" % L)


def _decode_vt(kc, vc, n0, steps, scale):
    q, k, v, w, beta = (cuda(t) for t in steps)
    ws = P.alloc_workspace(P.path_decode_workspace_bytes(*kc.shape), kc.device)
    outs, lses = [], []
    for t in range(q.shape[0]):
        o, lse = P.path_decode_step(q[t], k[t], v[t], w[t], beta[t], kc, vc, n0 + t, scale=scale, lse=True,
                                    workspace=ws, value_transport=True)
        outs.append(o)
        lses.append(lse)
    torch.cuda.synchronize()
    assert P.path_get_status(ws) == P.PATH_OK
    return torch.stack(outs), torch.stack(lses)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128), ("bf16", 16)])
def test_decode_vt_vs_oracle(dtype, d):
    """A cache of transported keys and values (both sampled directly), 10 steps with both caches
    transported in place."""
    B, H, n0, T = 2, 2, 400, 10
    kc, vc = inputs.make_decode_cache(B, H, n0, d, n0 + T, dtype, seed=8)
    steps = inputs.make_decode_steps(B, H, d, T, dtype, seed=8)
    scale = d ** -0.5
    k0, v0 = kc.clone(), vc.clone()
    kcg, vcg = kc.cuda(), vc.cuda()
    o, lse = _decode_vt(kcg, vcg, n0, steps, scale)
    f = inputs.f64
    for b in range(B):
        for h in range(H):
            o_ref, lse_ref, kc_ref, vc_ref = orc.path_decode(
                f(k0[b, h, :n0]), f(v0[b, h, :n0]), *(f(t[:, b, h]) for t in steps[:4]), f(steps[4][:, b, h]),
                scale, value_transport=True)
            check(to_np(o[:, b, h]), o_ref, kc.dtype, "decode vt b%d h%d" % (b, h))
            check_lse(to_np(lse[:, b, h]), lse_ref, kc.dtype, "decode vt lse")
            for got, ref in ((kcg[b, h], kc_ref), (vcg[b, h], vc_ref)):
                err = np.abs(to_np(got) - ref)
                if dtype == "f32":
                    assert err.max() <= 1e-5
                else:  # one bf16 rounding per step: at most T half-ulps of drift per element
                    assert np.all(err <= T * 2.0 ** -8 * np.abs(ref).max(axis=1, keepdims=True))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_vt_from_empty_equals_fwd_vt(dtype):
    """Token by token from empty caches (both transported in place) reproduces the value-transport
    forward, and the value cache left behind is the prefill hand-off applied to v."""
    B, H, L, d = 1, 2, 160, 64
    x = inputs.make_fwd(B, H, L, d, dtype, seed=520)
    o_fwd, _ = _vt_fwd(x)
    kc = torch.zeros((B, H, L, d), dtype=x.q.dtype, device="cuda")
    vc = torch.zeros_like(kc)
    steps = [t.permute(2, 0, 1, 3).contiguous() for t in (x.q, x.k, x.v, x.w)]
    steps.append(x.beta.permute(2, 0, 1).contiguous())
    o_dec, _ = _decode_vt(kc, vc, 0, steps, x.scale)
    o_dec = o_dec.permute(1, 2, 0, 3)
    diff = float((o_dec.float() - o_fwd.float()).abs().max())
    assert diff <= (2e-5 if dtype == "f32" else 3e-2), diff
    # the hand-off computes the same transported value cache from v in one pass; both caches against
    # the oracle's H_{L-1} ... H_{j+1} v_j (the decode cache is rounded to the cache dtype once per
    # step, the hand-off a few times in all)
    vh = P.path_prefill_kcache(cuda(x.v), cuda(x.w), cuda(x.beta))
    torch.cuda.synchronize()
    f = inputs.f64
    for h in range(H):
        _, _, _, vc_ref = orc.path_decode(np.zeros((0, d)), np.zeros((0, d)),
                                          *(f(t[0, h]) for t in (x.q, x.k, x.v, x.w, x.beta)), x.scale,
                                          value_transport=True)
        row = np.abs(vc_ref).max(axis=1, keepdims=True)
        e_dec = np.abs(to_np(vc[0, h]) - vc_ref)
        e_hand = np.abs(to_np(vh[0, h]) - vc_ref)
        if dtype == "f32":
            assert e_dec.max() <= 1e-4 and e_hand.max() <= 1e-4
        else:
            assert np.all(e_dec <= L * 2.0 ** -8 * row)
            assert np.all(e_hand <= 4 * 2.0 ** -8 * row + 1e-6)


def test_decode_vt_32k_sampled_heads():
    """B64 H12 d128 bf16 at a 32768-token cache, 16 steps with both caches transported; the oracle
    replays 2 sampled heads."""
    cfg = inputs.DECODE_CONFIGS["decode32k_bf16"]
    T = 16
    n_max = cfg.n0 + T
    kc, vc = inputs.make_decode_cache(cfg.B, cfg.H, cfg.n0, cfg.d, n_max, cfg.dtype, cfg.seed)
    steps = [t[:T] for t in inputs.make_decode_steps(cfg.B, cfg.H, cfg.d, cfg.steps, cfg.dtype, cfg.seed)]
    kcg, vcg = kc.cuda(), vc.cuda()
    del kc, vc
    scale = cfg.d ** -0.5
    o, lse = _decode_vt(kcg, vcg, cfg.n0, steps, scale)
    heads = [5, cfg.B * cfg.H - 2]
    kh, vh = inputs.make_decode_cache(cfg.B, cfg.H, cfg.n0, cfg.d, n_max, cfg.dtype, cfg.seed, heads=heads)
    f = inputs.f64
    for i, bh in enumerate(heads):
        b, h = divmod(bh, cfg.H)
        o_ref, lse_ref, _, _ = orc.path_decode(f(kh[i]), f(vh[i]), *(f(t[:, b, h]) for t in steps[:4]),
                                               f(steps[4][:, b, h]), scale, value_transport=True)
        check(to_np(o[:, b, h]), o_ref, torch.bfloat16, "decode32k vt head %d" % bh)
        check_lse(to_np(lse[:, b, h]), lse_ref, torch.bfloat16, "decode32k vt lse head %d" % bh)
