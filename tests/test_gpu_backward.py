"""GPU backward parity: path_attn_bwd (through the C ABI) against the fp64 oracle's gradients.

Every gradient (dq, dk, dv, dw, dbeta, and dlog f with PaTH-FoX forget gates) is compared element
by element with oracle.path_attn_bwd on the same dtype-rounded inputs and the same dO; o and lse
come from the GPU forward, as a caller would pass them.  Cases cover one chunk (no chunk pairs),
ragged last chunks, beta = 0 / beta = 2 positions, d = 16..128, both dtypes, and two whole heads
sampled from the 760M-shaped B8 H12 L4096 d128 bf16 workload that bench.py times.

Tolerances, as fractions of the largest magnitude of each reference gradient (every gradient has
its own scale; the scale is floored at 1e-3 for gradients that vanish, e.g. dq at L = 1):
  fp32: max abs error <= 1e-4.  The kernels add O(L) fp32 terms per output and walk at most 64
        transitions per chunk, so rounding stays near 1e-6 of the scale; 1e-4 leaves room for the
        approximate exponential and the forward's fp32 lse.
  bf16: max abs error <= 3e-2, mean abs error <= 3e-3.  Gradients are stored in bf16 (2^-9
        relative), and Delta_i = dO_i . o_i is formed from the forward's bf16 output o, whose own
        error (up to 2e-2) moves every dS_ij of the row by p_ij times the Delta error.
"""
import numpy as np
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import cuda, to_np
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dw", "dbeta")
TOL = {torch.float32: (1e-4, None), torch.bfloat16: (3e-2, 3e-3)}


def _dO(shape, dtype, seed):
    g = torch.Generator().manual_seed(1000 + seed)
    return torch.randn(shape, generator=g).to(dtype)


def _gpu_bwd(x: inputs.FwdInputs, dO: torch.Tensor):
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    lf = cuda(x.log_f)
    # the bf16 forward runs at d = 64 and 128; below that a caller forms o and lse in fp32 from the
    # same (bf16) values and rounds o to bf16, as done here
    fargs = args if (x.q.dtype == torch.float32 or x.q.shape[-1] >= 64) else [a.float() for a in args[:4]] + args[4:]
    if lf is not None:
        o, lse = P.path_attn_fwd_fox(*fargs, lf, scale=x.scale, lse=True)
    else:
        o, lse = P.path_attn_fwd(*fargs, scale=x.scale, lse=True)
    o = o.to(x.q.dtype)
    B, H, L, d = x.q.shape
    ws = P.alloc_workspace(P.path_attn_bwd_workspace_bytes(B, H, L, d, x.q.dtype), "cuda")
    g = P.path_attn_bwd(*args, o, lse, cuda(dO), log_f=lf, scale=x.scale, workspace=ws)
    torch.cuda.synchronize()
    assert P.path_get_status(ws) == P.PATH_OK
    return g


def _oracle(x: inputs.FwdInputs, dO, heads=None):
    f = inputs.f64
    ts = [x.q, x.k, x.v, x.w, x.beta, dO] + ([] if x.log_f is None else [x.log_f])
    if heads is None:
        ts = [f(t) for t in ts]
    else:  # slice before widening: a whole 760M-shaped tensor in fp64 is 3 GB
        ts = [np.stack([f(t[b, h]) for (b, h) in heads]) for t in ts]
    q, k, v, w, beta, g = ts[:6]
    lf = ts[6] if len(ts) > 6 else None
    return orc.path_attn_bwd(q, k, v, w, beta, g, log_f=lf, scale=x.scale)


def _compare(got, ref, dtype, what):
    tmax, tmean = TOL[dtype]
    names = NAMES + (("dlog_f",) if "dlog_f" in ref else ())
    errs = {}
    for n in names:
        g = np.asarray(got[n], np.float64)
        r = np.asarray(ref[n], np.float64)
        assert g.shape == r.shape, (n, g.shape, r.shape)
        assert np.all(np.isfinite(g)), "%s %s: non-finite" % (what, n)
        scale = max(float(np.abs(r).max()), 1e-3)  # a gradient that vanishes exactly is held to 1e-3 absolute scale
        err = np.abs(g - r)
        errs[n] = float(err.max()) / scale
        assert errs[n] <= tmax, "%s %s: max abs err %.3g of max |ref| %.3g > %.1g" % (what, n, errs[n], scale, tmax)
        if tmean is not None:
            assert float(err.mean()) / scale <= tmean, "%s %s: mean abs err %.3g" % (what, n, err.mean() / scale)
    print("%s: max abs err / max |ref| %s" % (what, " ".join("%s %.2g" % kv for kv in errs.items())))
    return errs


def _case(x: inputs.FwdInputs, seed, what):
    dO = _dO(x.q.shape, x.q.dtype, seed)
    g = _gpu_bwd(x, dO)
    ref = _oracle(x, dO)
    got = {n: to_np(t) for n, t in g.items()}
    return _compare(got, ref, x.q.dtype, what)


@pytest.mark.parametrize("fox", [False, True])
def test_bwd_single_chunk_f32(fox):
    """L = 64 = one chunk: only the within-chunk walks and the diagonal block."""
    x = inputs.make_fwd(1, 1, 64, 16, "f32", seed=0, fox=fox)
    _case(x, 0, "tiny fox=%s" % fox)


@pytest.mark.parametrize("B,H,L,d,fox", [(1, 2, 200, 32, False), (2, 1, 129, 64, True), (1, 2, 300, 128, False),
                                         (1, 1, 300, 128, True)])
def test_bwd_f32_ragged(B, H, L, d, fox):
    """Several chunks with a ragged last chunk, beta = 0 and beta = 2 positions included."""
    x = inputs.make_fwd(B, H, L, d, "f32", seed=11 + L, beta_std=2.0, edge_frac=0.05, fox=fox)
    _case(x, L, "f32 B%d H%d L%d d%d fox=%s" % (B, H, L, d, fox))


@pytest.mark.parametrize("L", [2, 65])
def test_bwd_short_lengths(L):
    """Two tokens, and a second chunk of a single row."""
    x = inputs.make_fwd(2, 1, L, 16, "f32", seed=40 + L, fox=True)
    _case(x, 40 + L, "f32 L%d" % L)


def test_bwd_single_token():
    """L = 1: the lone key has probability 1, so dv = dO and dq = dk = 0 up to the fp32 cancellation in
    dO.v - dO.o (|dO.v| ~ 10 here, so 1e-5 absolute); no transition and no forget gate enters a logit,
    so dbeta, dw and dlog f vanish exactly."""
    x = inputs.make_fwd(2, 3, 1, 16, "f32", seed=41, fox=True)
    dO = _dO(x.q.shape, torch.float32, 41)
    g = _gpu_bwd(x, dO)
    np.testing.assert_allclose(to_np(g["dv"]), to_np(dO), rtol=0, atol=1e-6)
    assert float(g["dq"].abs().max()) <= 1e-5 and float(g["dk"].abs().max()) <= 1e-5
    for n in ("dbeta", "dw", "dlog_f"):
        assert float(g[n].abs().max()) == 0.0, n


def test_bwd_f32_beta_zero_is_attention_backward():
    """beta = 0: dq, dk, dv equal torch's causal SDPA backward (fp32 on the GPU), dw = 0."""
    x = inputs.make_fwd(1, 2, 190, 64, "f32", seed=21)
    x.beta.zero_()
    dO = _dO(x.q.shape, torch.float32, 21)
    g = _gpu_bwd(x, dO)
    tq, tk, tv = (cuda(t).clone().requires_grad_(True) for t in (x.q, x.k, x.v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=x.scale)
    o.backward(cuda(dO))
    for n, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        ref = t.grad.double()
        err = float((g[n].double() - ref).abs().max()) / float(ref.abs().max())
        assert err <= 1e-4, (n, err)
    assert float(g["dw"].abs().max()) == 0.0


def test_bwd_small_bf16_config():
    """The small bf16 workload (B2 H4 L1024 d64, 5 % / 5 % beta = 0 / 2 edge positions), every head."""
    x = inputs.FWD_CONFIGS["small_bf16"].make()
    _case(x, 1, "small_bf16")


@pytest.mark.parametrize("B,H,L,fox", [(2, 3, 517, False), (1, 2, 130, True)])
def test_bwd_bf16_d128_edge_betas(B, H, L, fox):
    """The tensor-core chains and sums (bf16, d = 128) with 5 % / 5 % beta = 0 / beta = 2 positions, a ragged
    last chunk, several heads and odd chunk counts (L = 517: 9 chunks, L = 130: 3), where chunk 0, which has no
    chain, is the one left unpaired."""
    x = inputs.make_fwd(B, H, L, 128, "bf16", seed=70 + L, beta_std=2.0, edge_frac=0.05, fox=fox)
    _case(x, 70 + L, "bf16 d128 edges B%d H%d L%d fox=%s" % (B, H, L, fox))


def test_bwd_bf16_fox_d128_ragged():
    x = inputs.make_fwd(1, 2, 333, 128, "bf16", seed=33, fox=True)
    _case(x, 33, "bf16 fox L333")


@pytest.mark.parametrize("B,H,L,d,fox", [(2, 1, 177, 64, True), (1, 2, 200, 32, True), (1, 2, 130, 16, False)])
def test_bwd_bf16_small_d_ragged(B, H, L, d, fox):
    """bf16 below d = 128 with ragged last chunks and beta = 0 / 2 positions: at d = 64 the within-chunk
    stage and the prep run their products on the tensor cores (mma.sync), at d = 16 and 32 on the
    CUDA cores."""
    x = inputs.make_fwd(B, H, L, d, "bf16", seed=90 + d, beta_std=2.0, edge_frac=0.05, fox=fox)
    _case(x, 90 + L, "bf16 B%d H%d L%d d%d fox=%s" % (B, H, L, d, fox))


@pytest.mark.parametrize("L,fox", [(64, True), (100, False), (1, True)])
def test_bwd_bf16_d128_one_or_two_chunks(L, fox):
    """bf16 d = 128 with one chunk (no chains: only the diagonal block and the within-chunk products) or
    two (one chain step and no inner chunk, so no chunk transition P_m enters)."""
    x = inputs.make_fwd(2, 2, L, 128, "bf16", seed=120 + L, beta_std=2.0, edge_frac=0.05, fox=fox)
    _case(x, 120 + L, "bf16 d128 L%d fox=%s" % (L, fox))


def test_bwd_760m_shaped_sampled_heads():
    """The bench's backward workload, B8 H12 L4096 d128 bf16, run whole; two heads (first and
    last) compared with the oracle over every position."""
    x = inputs.FWD_CONFIGS["path760m_bf16"].make()
    dO = _dO(x.q.shape, torch.bfloat16, 2)
    g = _gpu_bwd(x, dO)
    heads = [(0, 0), (7, 11)]
    ref = _oracle(x, dO, heads=heads)
    got = {n: np.stack([to_np(t[b, h]) for (b, h) in heads]) for n, t in g.items()}
    _compare(got, ref, torch.bfloat16, "760m sampled heads")


def test_bwd_fox16k_two_whole_heads():
    """The PaTH-FoX long-context workload, B1 H12 L16384 d128 bf16 (log f = logsigmoid(N(3,1))),
    backward run whole; heads 0 and 11 compared with the oracle over every position, dlog f
    included."""
    x = inputs.FWD_CONFIGS["fox16k_bf16"].make()
    dO = _dO(x.q.shape, torch.bfloat16, 16)
    g = _gpu_bwd(x, dO)
    heads = [(0, 0), (0, 11)]
    ref = _oracle(x, dO, heads=heads)
    got = {n: np.stack([to_np(t[b, h]) for (b, h) in heads]) for n, t in g.items()}
    _compare(got, ref, torch.bfloat16, "fox16k whole heads")
