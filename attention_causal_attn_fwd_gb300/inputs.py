"""Seeded synthetic inputs for PaTH attention, shared by the tests, the bench and the oracle runs.

This module holds no PaTH arithmetic: it only draws q, k, v, w, beta and log f
with the distributions of the workloads below, on a CPU ``torch.Generator`` so
that every machine sees identical values.  Values are sampled in fp32, w is
normalised to unit L2 norm in fp32, and q, k, v, w are then rounded to the
compute dtype.  beta and log f stay fp32.  The oracle reads the rounded values
(upcast to fp64), so both sides consume identical numbers.

Workloads (stand-ins for the 760M-parameter, 4K-context language-model setting
and the 16K-64K length-extrapolation setting of "Resumo Técnico: Atenção PaTH",
§4 "Modelagem de Linguagem (760M Parâmetros)"; no dataset or trained weight is
used):

=================  ==============================================================
tiny_f32           B1 H1 L64 d16 fp32; beta = 2 sigmoid(N(0,1)); seed 0
small_bf16         B2 H4 L1024 d64 bf16; beta = 2 sigmoid(N(0, std 2)), 5% of
                   positions forced to beta = 0 and 5% to beta = 2; seed 1
path760m_bf16      B8 H12 L4096 d128 bf16 (hidden 1536); beta = 2 sigmoid(N(0,1));
                   seed 2 — the headline forward workload
fox16k_bf16        B1 H12 L16384 d128 bf16 + log f = logsigmoid(N(3,1)); seed 3
fox64k_bf16        B1 H12 L65536 d128 bf16 + log f = logsigmoid(N(3,1)); seed 5
decode32k_bf16     B64 H12 d128 bf16; cache of 32768 Gaussian (already
                   transported) keys and values; 256 steps, each with fresh
                   q, k, v ~ N(0,1), unit w_t, beta_t = 2 sigmoid(N(0,1)); seed 4
=================  ==============================================================

ggd_bam_bias() draws the per-head relative-position tables of the GGD-BAM prior used
with path_attn_fwd_relbias (the bias is an input of that call, like log f).
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
from typing import Optional

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass
class FwdInputs:
    q: torch.Tensor          # [B, H, L, d] dtype
    k: torch.Tensor
    v: torch.Tensor
    w: torch.Tensor          # unit-norm rows (before rounding to dtype)
    beta: torch.Tensor       # [B, H, L] fp32
    log_f: Optional[torch.Tensor]  # [B, H, L] fp32 or None
    scale: float

    @property
    def shape(self):
        return tuple(self.q.shape)


@dataclasses.dataclass
class FwdConfig:
    name: str
    B: int
    H: int
    L: int
    d: int
    dtype: str
    seed: int
    beta_std: float = 1.0
    edge_frac: float = 0.0   # fraction forced to beta = 0, and the same fraction to beta = 2
    fox: bool = False

    def make(self, **over) -> FwdInputs:
        kw = dataclasses.asdict(self)
        kw.pop("name")
        kw.update(over)
        return make_fwd(**kw)

    @property
    def attn_flops(self) -> float:
        """Attention-equivalent FLOPs of one causal forward: 4 B H d L^2 / 2."""
        return 4.0 * self.B * self.H * self.d * self.L * self.L / 2.0


@dataclasses.dataclass
class DecodeConfig:
    name: str
    B: int
    H: int
    d: int
    n0: int
    steps: int
    dtype: str
    seed: int


FWD_CONFIGS = {
    "tiny_f32": FwdConfig("tiny_f32", 1, 1, 64, 16, "f32", 0),
    "small_bf16": FwdConfig("small_bf16", 2, 4, 1024, 64, "bf16", 1, beta_std=2.0, edge_frac=0.05),
    "path760m_bf16": FwdConfig("path760m_bf16", 8, 12, 4096, 128, "bf16", 2),
    "fox16k_bf16": FwdConfig("fox16k_bf16", 1, 12, 16384, 128, "bf16", 3, fox=True),
    # the long end of the pages' length-extrapolation range (16K-64K)
    "fox64k_bf16": FwdConfig("fox64k_bf16", 1, 12, 65536, 128, "bf16", 5, fox=True),
}
DECODE_CONFIGS = {
    "decode32k_bf16": DecodeConfig("decode32k_bf16", 64, 12, 128, 32768, 256, "bf16", 4),
}


def ggd_bam_bias(H: int, L: int, seed: int) -> torch.Tensor:
    """Per-head relative-position bias table [H, L] (fp32): entry (h, delta) is the GGD-BAM prior
    -|(j - i - mu_h) / alpha_h|^p_h at distance delta = i - j ("Resumo Técnico: Mecanismo de Atenção
    Bayesiana (BAM)", §"Solução Proposta: GGD-BAM").  Seeded per-head parameters: mu = 0, alpha_h
    log-uniform in [16, 512], p_h uniform in [0.5, 1.5] (heavy- to light-tailed around the Laplace /
    ALiBi case p = 1)."""
    g = _gen(seed)
    alpha = torch.exp(math.log(16.0) + (math.log(512.0) - math.log(16.0)) * torch.rand(H, generator=g, dtype=torch.float64))
    p = 0.5 + torch.rand(H, generator=g, dtype=torch.float64)
    delta = torch.arange(L, dtype=torch.float64)
    return (-(delta.view(1, L) / alpha.view(H, 1)).abs() ** p.view(H, 1)).float().contiguous()


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def make_fwd(B, H, L, d, dtype="bf16", seed=0, beta_std=1.0, edge_frac=0.0, fox=False) -> FwdInputs:
    """Draw one forward workload.  Draw order is fixed: q, k, v, w, beta, edge draws, log f."""
    g = _gen(seed)
    dt = DTYPES[dtype]
    shape = (B, H, L, d)
    q = torch.randn(shape, generator=g)
    k = torch.randn(shape, generator=g)
    v = torch.randn(shape, generator=g)
    w = _unit_rows(torch.randn(shape, generator=g))
    beta = 2.0 * torch.sigmoid(beta_std * torch.randn((B, H, L), generator=g))
    if edge_frac > 0:
        u = torch.rand((B, H, L), generator=g)
        beta = torch.where(u < edge_frac, torch.zeros_like(beta), beta)
        beta = torch.where((u >= edge_frac) & (u < 2 * edge_frac), torch.full_like(beta, 2.0), beta)
    log_f = None
    if fox:
        log_f = torch.nn.functional.logsigmoid(3.0 + torch.randn((B, H, L), generator=g))
    return FwdInputs(q.to(dt), k.to(dt), v.to(dt), w.to(dt), beta.float().contiguous(),
                     None if log_f is None else log_f.float().contiguous(), 1.0 / math.sqrt(d))


def make_decode_cache(B, H, n0, d, n_max, dtype="bf16", seed=4, heads=None, threads=16):
    """Prefilled caches [B, H, n_max, d]: rows < n0 ~ N(0,1) (keys taken as already
    transported), rows >= n0 zero.  Each head draws from its own generator
    (seed, head), so a subset of heads can be regenerated alone: with ``heads``
    (list of flat b*H+h) only those heads are returned, as [len(heads), n0, d]
    pairs (k, v).
    """
    dt = DTYPES[dtype]

    def one(bh):
        g = _gen(seed * 1_000_003 + 7919 * (bh + 1))
        kk = torch.randn((n0, d), generator=g).to(dt)
        vv = torch.randn((n0, d), generator=g).to(dt)
        return kk, vv

    if heads is not None:
        ks, vs = zip(*[one(int(h)) for h in heads])
        return torch.stack(ks), torch.stack(vs)
    kc = torch.zeros((B, H, n_max, d), dtype=dt)
    vc = torch.zeros((B, H, n_max, d), dtype=dt)
    kf = kc.view(B * H, n_max, d)
    vf = vc.view(B * H, n_max, d)

    def fill(bh):
        kk, vv = one(bh)
        kf[bh, :n0] = kk
        vf[bh, :n0] = vv

    with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, range(B * H)))
    return kc, vc


def make_decode_steps(B, H, d, T, dtype="bf16", seed=4):
    """Per-step decode inputs: q, k, v, w [T, B, H, d] (w unit-norm), beta [T, B, H] fp32."""
    g = _gen(seed * 1_000_003 + 1)
    dt = DTYPES[dtype]
    shape = (T, B, H, d)
    q = torch.randn(shape, generator=g)
    k = torch.randn(shape, generator=g)
    v = torch.randn(shape, generator=g)
    w = _unit_rows(torch.randn(shape, generator=g))
    beta = 2.0 * torch.sigmoid(torch.randn((T, B, H), generator=g))
    return q.to(dt), k.to(dt), v.to(dt), w.to(dt), beta.float().contiguous()


def f64(t: torch.Tensor):
    """Upcast a (rounded) input tensor to an fp64 numpy array for the oracle."""
    return t.detach().to("cpu", torch.float64).numpy()
