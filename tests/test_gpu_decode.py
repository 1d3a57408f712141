"""GPU decode parity: path_decode_step / path_kcache_update (through the C ABI) against the fp64
decode oracle, decode-from-empty = prefill, and the full-size 32K-cache decode on sampled heads."""
import numpy as np
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import check, check_lse, cuda, to_np
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _run_decode(kc, vc, n0, steps, scale):
    q, k, v, w, beta = (cuda(t) for t in steps)
    T = q.shape[0]
    ws = P.alloc_workspace(P.path_decode_workspace_bytes(kc.shape[0], kc.shape[1], kc.shape[2], kc.shape[3]),
                           kc.device)
    outs, lses = [], []
    for t in range(T):
        o, lse = P.path_decode_step(q[t], k[t], v[t], w[t], beta[t], kc, vc, n0 + t, scale=scale, lse=True,
                                    workspace=ws)
        outs.append(o)
        lses.append(lse)
    torch.cuda.synchronize()
    assert P.path_get_status(ws) == P.PATH_OK
    return torch.stack(outs), torch.stack(lses)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("f32", 128), ("bf16", 128), ("bf16", 64), ("bf16", 16)])
def test_decode_small_vs_oracle(dtype, d):
    B, H, n0, T = 2, 3, 300, 12
    kc, vc = inputs.make_decode_cache(B, H, n0, d, n0 + T, dtype, seed=5)
    steps = inputs.make_decode_steps(B, H, d, T, dtype, seed=5)
    scale = d ** -0.5
    kc_ref0, vc_ref0 = kc.clone(), vc.clone()
    kcg, vcg = kc.cuda(), vc.cuda()
    o, lse = _run_decode(kcg, vcg, n0, steps, scale)
    f = inputs.f64
    for b in range(B):
        for h in range(H):
            o_ref, lse_ref, kc_ref, vc_ref = orc.path_decode(
                f(kc_ref0[b, h, :n0]), f(vc_ref0[b, h, :n0]), *(f(t[:, b, h]) for t in steps[:4]),
                f(steps[4][:, b, h]), scale)
            check(to_np(o[:, b, h]), o_ref, kc.dtype, "decode o b%d h%d" % (b, h))
            check_lse(to_np(lse[:, b, h]), lse_ref, kc.dtype, "decode lse")
            err = np.abs(to_np(kcg[b, h]) - kc_ref)
            if dtype == "f32":
                assert err.max() <= 1e-5
            else:  # the bf16 cache is rounded once per step: at most T half-ulps of drift per element
                bound = T * 2.0 ** -8 * np.abs(kc_ref).max(axis=1, keepdims=True)
                assert np.all(err <= bound), float((err - bound).max())
            assert np.array_equal(to_np(vcg[b, h]), vc_ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_from_empty_cache_equals_prefill(dtype):
    """§3 "Inferência": token-by-token decode with in-place key updates reproduces the forward."""
    B, H, L, d = 1, 2, 150, 64
    x = inputs.make_fwd(B, H, L, d, dtype, seed=21)
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    o_fwd = P.path_attn_fwd(*args, scale=x.scale)
    kc = torch.zeros((B, H, L, d), dtype=x.q.dtype, device="cuda")
    vc = torch.zeros_like(kc)
    steps = [t.transpose(0, 2).transpose(1, 2).contiguous() for t in (x.q, x.k, x.v, x.w)]  # [L, B, H, d]
    steps.append(x.beta.permute(2, 0, 1).contiguous())
    o_dec, _ = _run_decode(kc, vc, 0, steps, x.scale)
    o_dec = o_dec.permute(1, 2, 0, 3)
    o_ref, _ = orc.path_attn(*(inputs.f64(t) for t in (x.q, x.k, x.v, x.w, x.beta)), scale=x.scale)
    check(to_np(o_dec), o_ref, x.q.dtype, "decode-from-empty vs oracle prefill")
    diff = float((o_dec.float() - o_fwd.float()).abs().max())
    assert diff <= (2e-5 if dtype == "f32" else 3e-2), diff


@pytest.mark.parametrize("dtype,d", [("f32", 128), ("bf16", 128), ("bf16", 32)])
def test_kcache_update_vs_oracle(dtype, d):
    B, H, n_max, n = 2, 2, 700, 650
    kc, _ = inputs.make_decode_cache(B, H, n, d, n_max, dtype, seed=6)
    _, _, _, w, beta = inputs.make_decode_steps(B, H, d, 1, dtype, seed=6)
    kcg = kc.cuda()
    P.path_kcache_update(kcg, n, w[0].cuda(), beta[0].cuda())
    torch.cuda.synchronize()
    f = inputs.f64
    for b in range(B):
        for h in range(H):
            ref = orc.kcache_update(f(kc[b, h, :n]), f(w[0, b, h]), float(beta[0, b, h]))
            got = to_np(kcg[b, h, :n])
            if dtype == "f32":
                assert np.abs(got - ref).max() <= 1e-5
            else:  # fp32 arithmetic, one rounding to bf16: within one bf16 ulp
                assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)
            assert torch.equal(kcg[b, h, n:], kc[b, h, n:].cuda())  # rows >= n untouched


def test_decode32k_full_size_sampled_heads():
    """B64 H12 d128 bf16, 32768-token cache, 256 steps on the GPU (the timed workload);
    the oracle replays 3 sampled heads over all 256 steps from the same cache."""
    cfg = inputs.DECODE_CONFIGS["decode32k_bf16"]
    n_max = cfg.n0 + cfg.steps
    kc, vc = inputs.make_decode_cache(cfg.B, cfg.H, cfg.n0, cfg.d, n_max, cfg.dtype, cfg.seed)
    steps = inputs.make_decode_steps(cfg.B, cfg.H, cfg.d, cfg.steps, cfg.dtype, cfg.seed)
    kcg, vcg = kc.cuda(), vc.cuda()
    del kc, vc
    scale = cfg.d ** -0.5
    o, lse = _run_decode(kcg, vcg, cfg.n0, steps, scale)
    assert torch.isfinite(o).all()
    heads = [0, 377, cfg.B * cfg.H - 1]
    kh, vh = inputs.make_decode_cache(cfg.B, cfg.H, cfg.n0, cfg.d, n_max, cfg.dtype, cfg.seed, heads=heads)
    f = inputs.f64
    for i, bh in enumerate(heads):
        b, h = divmod(bh, cfg.H)
        o_ref, lse_ref, _, _ = orc.path_decode(f(kh[i]), f(vh[i]), *(f(t[:, b, h]) for t in steps[:4]),
                                               f(steps[4][:, b, h]), scale)
        check(to_np(o[:, b, h]), o_ref, torch.bfloat16, "decode32k head %d" % bh)
        check_lse(to_np(lse[:, b, h]), lse_ref, torch.bfloat16, "decode32k lse head %d" % bh)


def test_kv_cache_checkpoint_and_resume_is_bit_identical():
    """Checkpoint / resume ("Resumo Técnico: Atenção PaTH", §3 "Inferência": the transported key cache
    and the value cache are the whole decoding state).  Decode 5 steps, copy both caches to host
    memory, then continue 4 more steps twice: on the live caches, and on fresh device caches restored
    from the host copy.  The continuations must agree bit for bit, outputs and caches."""
    B, H, d, n0, T1, T2 = 2, 3, 128, 1500, 5, 4
    kc, vc = inputs.make_decode_cache(B, H, n0, d, n0 + T1 + T2, "bf16", seed=44)
    steps = [t.cuda() for t in inputs.make_decode_steps(B, H, d, T1 + T2, "bf16", seed=44)]
    k, v = kc.cuda(), vc.cuda()
    for t in range(T1):
        P.path_decode_step(*(s[t] for s in steps), k, v, n0 + t)
    torch.cuda.synchronize()
    host_k, host_v = k.cpu(), v.cpu()  # the checkpoint
    live = [P.path_decode_step(*(s[t] for s in steps), k, v, n0 + t) for t in range(T1, T1 + T2)]
    k2, v2 = host_k.cuda(), host_v.cuda()  # resume on fresh buffers
    resumed = [P.path_decode_step(*(s[t] for s in steps), k2, v2, n0 + t) for t in range(T1, T1 + T2)]
    torch.cuda.synchronize()
    for a, b in zip(live, resumed):
        assert torch.equal(a, b)
    assert torch.equal(k, k2) and torch.equal(v, v2)
