"""GPU forward parity: path_attn_fwd / path_attn_fwd_fox (through the C ABI) against the fp64 oracle.

Cases follow the workloads of attention_causal_attn_fwd_gb300.inputs (tiny fp32, small bf16
with beta = 0 / beta = 2 edge positions, 760M-shaped L=4096 d=128, PaTH-FoX L=16384) plus
ragged lengths, single-token sequences, beta special values and determinism.
"""
import numpy as np
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import check, check_lse, cuda, to_np
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _workspace(x: inputs.FwdInputs):
    B, H, L, d = x.q.shape
    return P.alloc_workspace(P.path_attn_workspace_bytes(B, H, L, d, x.q.dtype), "cuda")


def _gpu_fwd(x: inputs.FwdInputs):
    """GPU forward through the C ABI; the workspace status word must read PATH_OK afterwards (no
    bounded wait, including a drain before exit, ran out)."""
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    ws = _workspace(x)
    if x.log_f is not None:
        o, lse = P.path_attn_fwd_fox(*args, cuda(x.log_f), scale=x.scale, lse=True, workspace=ws)
    else:
        o, lse = P.path_attn_fwd(*args, scale=x.scale, lse=True, workspace=ws)
    torch.cuda.synchronize()
    assert P.path_get_status(ws) == P.PATH_OK
    return o, lse


def _oracle(x: inputs.FwdInputs, heads=None, rows=None):
    """Oracle on all heads, or on (head, row) samples: heads = list of (b, h), rows = list of i."""
    f = inputs.f64
    lf = None if x.log_f is None else f(x.log_f)
    if heads is None:
        return orc.path_attn(f(x.q), f(x.k), f(x.v), f(x.w), f(x.beta), lf, x.scale)
    sel = lambda t: np.stack([t[b, h] for (b, h) in heads])
    qs, ks, vs, ws, bs = (sel(f(t)) for t in (x.q, x.k, x.v, x.w, x.beta))
    ls = None if lf is None else np.stack([lf[b, h] for (b, h) in heads])
    L = x.q.shape[2]
    flat = [hi * L + i for hi in range(len(heads)) for i in rows]
    return orc.path_attn(qs, ks, vs, ws, bs, ls, x.scale, rows=flat)


def _full_case(x, what):
    o, lse = _gpu_fwd(x)
    o_ref, lse_ref = _oracle(x)
    check(to_np(o), o_ref, x.q.dtype, what)
    check_lse(to_np(lse), lse_ref, x.q.dtype, what)


def test_tiny_f32_config():
    _full_case(inputs.FWD_CONFIGS["tiny_f32"].make(), "tiny_f32")


def test_small_bf16_config():
    _full_case(inputs.FWD_CONFIGS["small_bf16"].make(), "small_bf16")


@pytest.mark.parametrize("dtype,B,H,L,d", [
    ("f32", 1, 2, 77, 32), ("f32", 2, 1, 1, 64), ("f32", 1, 1, 200, 128), ("f32", 1, 1, 50, 16),
    ("bf16", 1, 2, 300, 128), ("bf16", 1, 1, 1, 64), ("bf16", 2, 2, 129, 64), ("bf16", 1, 1, 257, 128),
    ("bf16", 1, 1, 640, 128),
])
def test_ragged_shapes(dtype, B, H, L, d):
    x = inputs.make_fwd(B, H, L, d, dtype, seed=100 + L + d, edge_frac=0.05)
    _full_case(x, "ragged %s %s" % (dtype, (B, H, L, d)))


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
@pytest.mark.parametrize("beta_kind", ["zero", "two", "half_zero"])
def test_beta_special_values(dtype, d, beta_kind):
    x = inputs.make_fwd(1, 2, 260, d, dtype, seed=7)
    if beta_kind == "zero":
        x.beta.zero_()
    elif beta_kind == "two":
        x.beta.fill_(2.0)
    else:
        x.beta[..., ::2] = 0.0
    _full_case(x, "beta %s" % beta_kind)


@pytest.mark.parametrize("dtype,L,d", [("f32", 100, 32), ("bf16", 300, 128), ("bf16", 200, 64)])
def test_fox_small(dtype, L, d):
    x = inputs.make_fwd(1, 2, L, d, dtype, seed=11, fox=True)
    _full_case(x, "fox %s" % dtype)


@pytest.mark.parametrize("dtype,d", [("f32", 32), ("bf16", 128)])
def test_fox_zero_gates_equal_plain(dtype, d):
    x = inputs.make_fwd(1, 2, 200, d, dtype, seed=12)
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    o1 = P.path_attn_fwd(*args, scale=x.scale)
    o2 = P.path_attn_fwd_fox(*args, torch.zeros_like(args[4]), scale=x.scale)
    torch.cuda.synchronize()
    assert float((o1.float() - o2.float()).abs().max()) <= (1e-6 if dtype == "f32" else 1e-2)


def test_deterministic():
    x = inputs.make_fwd(1, 2, 300, 128, "bf16", seed=13)
    o1, l1 = _gpu_fwd(x)
    o2, l2 = _gpu_fwd(x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _sampled_rows(L, rng, n=10):
    rows = {0, 1, 63, 64, 127, 128, L - 1, L // 2}
    rows |= set(int(i) for i in rng.integers(0, L, n))
    return sorted(r for r in rows if r < L)


def test_760m_shaped_full_size_sampled():
    """B8 H12 L4096 d128 bf16 (the timed workload): the whole forward on the GPU, sampled rows on the oracle."""
    cfg = inputs.FWD_CONFIGS["path760m_bf16"]
    x = cfg.make()
    o, lse = _gpu_fwd(x)
    rng = np.random.default_rng(0)
    heads = [(0, 0), (3, 7), (7, 11)]
    rows = _sampled_rows(cfg.L, rng)
    o_ref, lse_ref = _oracle(x, heads, rows)
    got = np.concatenate([to_np(o[b, h, rows]) for (b, h) in heads])
    got_lse = np.concatenate([to_np(lse[b, h, rows]) for (b, h) in heads])
    check(got, o_ref, torch.bfloat16, "path760m sampled")
    check_lse(got_lse, lse_ref, torch.bfloat16, "path760m sampled")
    assert torch.isfinite(o).all()


def test_fox_16k_full_size_sampled():
    """B1 H12 L16384 d128 bf16 PaTH-FoX: whole forward on the GPU, sampled rows on the oracle."""
    cfg = inputs.FWD_CONFIGS["fox16k_bf16"]
    x = cfg.make()
    o, lse = _gpu_fwd(x)
    rng = np.random.default_rng(1)
    heads = [(0, 0), (0, 5), (0, 11)]
    rows = _sampled_rows(cfg.L, rng, n=6)
    o_ref, lse_ref = _oracle(x, heads, rows)
    got = np.concatenate([to_np(o[b, h, rows]) for (b, h) in heads])
    got_lse = np.concatenate([to_np(lse[b, h, rows]) for (b, h) in heads])
    check(got, o_ref, torch.bfloat16, "fox16k sampled")
    check_lse(got_lse, lse_ref, torch.bfloat16, "fox16k sampled")
    assert torch.isfinite(o).all()


@pytest.mark.parametrize("L", [1000, 2048])
def test_fox_strong_gates_far_blocks_skipped(L):
    """Strong forget gates (log f = logsigmoid(N(0,1))) make every key more than a few hundred
    tokens away contribute exactly zero, so the scan stops early; every row must still match."""
    x = inputs.make_fwd(1, 3, L, 128, "bf16", seed=61, fox=True)
    g = torch.Generator().manual_seed(61)
    x.log_f = torch.nn.functional.logsigmoid(torch.randn(x.beta.shape, generator=g)).float()
    _full_case(x, "fox strong gates L=%d" % L)


def test_fox_64k_full_size_sampled():
    """B1 H12 L65536 d128 bf16 PaTH-FoX (the long end of the pages' 16K-64K extrapolation range):
    whole forward on the GPU, sampled rows on the oracle."""
    cfg = inputs.FWD_CONFIGS["fox64k_bf16"]
    x = cfg.make()
    o, lse = _gpu_fwd(x)
    rng = np.random.default_rng(2)
    heads = [(0, 0), (0, 11)]
    rows = _sampled_rows(cfg.L, rng, n=4)
    o_ref, lse_ref = _oracle(x, heads, rows)
    got = np.concatenate([to_np(o[b, h, rows]) for (b, h) in heads])
    got_lse = np.concatenate([to_np(lse[b, h, rows]) for (b, h) in heads])
    check(got, o_ref, torch.bfloat16, "fox64k sampled")
    check_lse(got_lse, lse_ref, torch.bfloat16, "fox64k sampled")
    assert torch.isfinite(o).all()


@pytest.mark.parametrize("dtype,d,beta_zero", [("bf16", 128, True), ("bf16", 64, True), ("f32", 32, True),
                                               ("bf16", 128, False)])
def test_alibi_as_constant_forget_gate(dtype, d, beta_zero):
    """A per-head ALiBi bias -slope (i - j) is the FoX bias with log f_s = -slope for every s.  With
    beta = 0 the result must be textbook ALiBi attention (fp64 SDPA with the explicit bias matrix,
    independent of the PaTH oracle); with random beta it is PaTH + ALiBi, checked on the oracle."""
    B, H, L = 1, 4, 700
    x = inputs.make_fwd(B, H, L, d, dtype, seed=71)
    if beta_zero:
        x.beta.zero_()
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)])
    x.log_f = (-slopes).view(1, H, 1).expand(B, H, L).contiguous().float()
    o, lse = _gpu_fwd(x)
    f = inputs.f64
    if beta_zero:
        i = torch.arange(L, dtype=torch.float64)
        rel = i.view(L, 1) - i.view(1, L)
        bias = torch.where(rel >= 0, -slopes.double().view(H, 1, 1) * rel, torch.tensor(float("-inf"), dtype=torch.float64))
        qd, kd, vd = (t.double() for t in (x.q, x.k, x.v))
        ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=bias.unsqueeze(0), scale=x.scale)
        check(to_np(o), ref.numpy(), x.q.dtype, "alibi %s d%d" % (dtype, d))
    else:
        o_ref, lse_ref = _oracle(x)
        check(to_np(o), o_ref, x.q.dtype, "PaTH + alibi")
        check_lse(to_np(lse), lse_ref, x.q.dtype, "PaTH + alibi")


def _relbias_case(x, rel):
    """GPU relative-bias forward against the oracle (table expanded over the batch)."""
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    ws = _workspace(x)
    o, lse = P.path_attn_fwd_relbias(*args, cuda(rel), scale=x.scale, lse=True, workspace=ws)
    torch.cuda.synchronize()
    assert P.path_get_status(ws) == P.PATH_OK
    B = x.q.shape[0]
    f = inputs.f64
    rb = np.broadcast_to(f(rel)[None], x.beta.shape).copy()
    return o, lse, rb


@pytest.mark.parametrize("dtype,B,H,L,d", [("bf16", 2, 3, 300, 128), ("bf16", 1, 2, 129, 64), ("bf16", 1, 1, 1, 128),
                                           ("f32", 1, 2, 150, 32), ("f32", 2, 1, 77, 64)])
def test_relbias_ggd_bam_vs_oracle(dtype, B, H, L, d):
    """PaTH + GGD-BAM relative-position prior (random beta, ragged L) against the oracle."""
    x = inputs.make_fwd(B, H, L, d, dtype, seed=91 + L, edge_frac=0.05)
    rel = inputs.ggd_bam_bias(H, L, seed=91)
    o, lse, rb = _relbias_case(x, rel)
    f = inputs.f64
    o_ref, lse_ref = orc.path_attn(f(x.q), f(x.k), f(x.v), f(x.w), f(x.beta), scale=x.scale, rel_bias=rb)
    check(to_np(o), o_ref, x.q.dtype, "relbias %s %s" % (dtype, (B, H, L, d)))
    check_lse(to_np(lse), lse_ref, x.q.dtype, "relbias lse")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_relbias_with_beta_zero_is_textbook_ggd_bam(dtype, d):
    """beta = 0: plain softmax attention with the GGD-BAM bias matrix (fp64 SDPA, independent of the
    PaTH oracle)."""
    B, H, L = 1, 3, 600
    x = inputs.make_fwd(B, H, L, d, dtype, seed=92)
    x.beta.zero_()
    rel = inputs.ggd_bam_bias(H, L, seed=92)
    o, _, _ = _relbias_case(x, rel)
    i = torch.arange(L)
    delta = (i.view(L, 1) - i.view(1, L)).clamp(min=0)
    bias = torch.where(i.view(L, 1) >= i.view(1, L), rel.double()[:, delta], torch.tensor(float("-inf"), dtype=torch.float64))
    ref = torch.nn.functional.scaled_dot_product_attention(*(t.double() for t in (x.q, x.k, x.v)),
                                                           attn_mask=bias.unsqueeze(0), scale=x.scale)
    check(to_np(o), ref.numpy(), x.q.dtype, "ggd-bam beta=0 %s" % dtype)


def test_relbias_linear_table_equals_fox_constant_gates():
    """An ALiBi table -slope * delta through the relative-bias path equals constant forget gates through
    the FoX path (two kernels, one operator)."""
    B, H, L, d = 1, 2, 520, 128
    x = inputs.make_fwd(B, H, L, d, "bf16", seed=93)
    slopes = torch.tensor([0.01, 0.05])
    rel = (-slopes.view(H, 1) * torch.arange(L, dtype=torch.float32).view(1, L)).contiguous()
    o1, _, _ = _relbias_case(x, rel)
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    lf = (-slopes).view(1, H, 1).expand(B, H, L).contiguous().float()
    o2 = P.path_attn_fwd_fox(*args, cuda(lf), scale=x.scale)
    torch.cuda.synchronize()
    assert float((o1.float() - o2.float()).abs().max()) <= 2e-2
