"""GPU forward at the workloads' full sizes, compared with the fp64 oracle on whole heads, and the
PaTH-FoX far-block stop checked for bit-identical results against visiting every block.

The oracle walks every query of a head through the transitions ("Resumo Técnico: Atenção PaTH",
§2 "Mecanismo Central"), so whole heads at L = 4096 and L = 16384 take seconds each on the host
cores; the GPU runs the whole batch.
"""
import numpy as np
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import check, check_lse, cuda, to_np
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _run(x, fox_skip=True):
    """Forward through the C ABI with the FoX far-block stop on or off; returns o, lse and the
    number of (query tile, key block) pairs visited."""
    B, H, L, d = x.q.shape
    ws = P.alloc_workspace(P.path_attn_workspace_bytes(B, H, L, d, x.q.dtype), "cuda")
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    P.path_debug_set_fox_skip(fox_skip)
    try:
        if x.log_f is None:
            o, lse = P.path_attn_fwd(*args, scale=x.scale, lse=True, workspace=ws)
        else:
            o, lse = P.path_attn_fwd_fox(*args, cuda(x.log_f), scale=x.scale, lse=True, workspace=ws)
        torch.cuda.synchronize()
        assert P.path_get_status(ws) == P.PATH_OK
        visited = P.path_fwd_visited_blocks(ws)
    finally:
        P.path_debug_set_fox_skip(True)
    return o, lse, visited


def _pairs(B, H, L):
    nt = -(-L // 128)
    return B * H * nt * (nt + 1) // 2


def _whole_heads(x, o, lse, heads, what):
    f = inputs.f64
    sel = lambda t: np.stack([t[b, h] for (b, h) in heads])
    args = [sel(f(t)) for t in (x.q, x.k, x.v, x.w, x.beta)]
    lf = None if x.log_f is None else sel(f(x.log_f))
    o_ref, lse_ref = orc.path_attn(*args, lf, x.scale)
    got = np.stack([to_np(o[b, h]) for (b, h) in heads])
    got_lse = np.stack([to_np(lse[b, h]) for (b, h) in heads])
    mx, mean = check(got, o_ref, x.q.dtype, what)
    check_lse(got_lse, lse_ref, x.q.dtype, what)
    return mx, mean


def test_760m_shaped_twelve_whole_heads():
    """B8 H12 L4096 d128 bf16, the timed workload: every row of 12 heads (one or two per batch entry,
    every head index once) against the oracle, and every (tile, block) pair visited."""
    cfg = inputs.FWD_CONFIGS["path760m_bf16"]
    x = cfg.make()
    o, lse, visited = _run(x)
    assert visited == _pairs(cfg.B, cfg.H, cfg.L)
    heads = [(h % cfg.B, h) for h in range(cfg.H)]
    _whole_heads(x, o, lse, heads, "path760m whole heads")
    assert torch.isfinite(o).all()


def test_fox_16k_two_whole_heads():
    """B1 H12 L16384 d128 bf16 PaTH-FoX: every row of heads 0 and 11 against the oracle."""
    cfg = inputs.FWD_CONFIGS["fox16k_bf16"]
    x = cfg.make()
    o, lse, visited = _run(x)
    assert 0 < visited <= _pairs(cfg.B, cfg.H, cfg.L)
    _whole_heads(x, o, lse, [(0, 0), (0, 11)], "fox16k whole heads")


def _strong_gates(L, H=3, seed=61):
    x = inputs.make_fwd(1, H, L, 128, "bf16", seed=seed, fox=True)
    g = torch.Generator().manual_seed(seed)
    x.log_f = torch.nn.functional.logsigmoid(torch.randn(x.beta.shape, generator=g)).float()
    return x


@pytest.mark.parametrize("case", ["fox16k", "strong_gates_2048", "strong_gates_700"])
def test_fox_far_block_stop_is_bit_identical(case):
    """The far-block stop skips a block only when every weight left of it is exactly 0 in fp32
    (preconditions beta in [0, 2], unit w, log f <= 0, all met by these inputs), so o and lse must be
    bit-identical to a run that visits every block, which must visit the full causal triangle."""
    if case == "fox16k":
        x = inputs.FWD_CONFIGS["fox16k_bf16"].make()
    else:
        x = _strong_gates(int(case.rsplit("_", 1)[1]))
    B, H, L, _ = x.q.shape
    o1, l1, v1 = _run(x, fox_skip=True)
    o2, l2, v2 = _run(x, fox_skip=False)
    assert v2 == _pairs(B, H, L)
    assert v1 <= v2
    if case != "fox16k":  # strong gates: most far blocks are skipped
        assert v1 < v2
    assert torch.equal(o1, o2), float((o1.float() - o2.float()).abs().max())
    assert torch.equal(l1, l2), float((l1 - l2).abs().max())
