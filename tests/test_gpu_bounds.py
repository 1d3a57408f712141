"""The bounds-checked build (-DPATH_DEBUG_BOUNDS) on small odd shapes: every plain global load and
store of the tensor-core forward, the UT prep, decode (with and without value transport) and the
value-transport forward checks its index against its buffer and
would record PATH_ERR_BOUNDS in the workspace status word.  Every call here must leave the status
PATH_OK, and its outputs must equal the normal build's bit for bit (the checks change no
arithmetic).  This stands in for the memory checker, which this environment does not offer."""
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import build as B
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    normal = P.load()
    checked = P.load(B.build(variant="debug_bounds"))
    yield normal, checked
    P._lib = normal


def _with(lib, fn):
    saved = P._lib
    P._lib = lib
    try:
        return fn()
    finally:
        P._lib = saved


@pytest.mark.parametrize("B_,H,L,d,mode", [(1, 1, 1, 128, "plain"), (1, 2, 77, 64, "plain"), (2, 1, 129, 128, "plain"),
                                           (1, 1, 300, 128, "fox"), (1, 2, 300, 64, "relbias"),
                                           (1, 1, 257, 128, "plain")])
def test_forward_bounds_checked(libs, B_, H, L, d, mode):
    normal, checked = libs
    x = inputs.make_fwd(B_, H, L, d, "bf16", seed=300 + L, fox=mode == "fox", edge_frac=0.05)
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]
    rel = cuda(inputs.ggd_bam_bias(H, L, seed=3)) if mode == "relbias" else None

    def run():
        ws = P.alloc_workspace(P.path_attn_workspace_bytes(B_, H, L, d, x.q.dtype), "cuda")
        if mode == "fox":
            o, lse = P.path_attn_fwd_fox(*args, cuda(x.log_f), scale=x.scale, lse=True, workspace=ws)
        elif mode == "relbias":
            o, lse = P.path_attn_fwd_relbias(*args, rel, scale=x.scale, lse=True, workspace=ws)
        else:
            o, lse = P.path_attn_fwd(*args, scale=x.scale, lse=True, workspace=ws)
        torch.cuda.synchronize()
        return o, lse, P.path_get_status(ws)

    o1, l1, st1 = _with(normal, run)
    o2, l2, st2 = _with(checked, run)
    assert st1 == P.PATH_OK and st2 == P.PATH_OK, (st1, st2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("dtype,B_,H,L,d,fox", [("bf16", 1, 1, 1, 128, False), ("bf16", 1, 2, 77, 64, True),
                                               ("f32", 2, 1, 129, 32, False), ("bf16", 1, 1, 300, 16, False)])
def test_value_transport_forward_bounds_checked(libs, dtype, B_, H, L, d, fox):
    normal, checked = libs
    x = inputs.make_fwd(B_, H, L, d, dtype, seed=400 + L, fox=fox, edge_frac=0.05)
    args = [cuda(t) for t in (x.q, x.k, x.v, x.w, x.beta)]

    def run():
        ws = P.alloc_workspace(P.load().path_attn_fwd_vt_workspace_bytes(B_, H, L, d, P._DT[x.q.dtype]), "cuda")
        o, lse = P.path_attn_fwd_vt(*args, log_f=cuda(x.log_f), scale=x.scale, lse=True, workspace=ws)
        torch.cuda.synchronize()
        return o, lse, P.path_get_status(ws)

    o1, l1, st1 = _with(normal, run)
    o2, l2, st2 = _with(checked, run)
    assert st1 == P.PATH_OK and st2 == P.PATH_OK, (st1, st2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d,n0,vt", [(128, 0, False), (64, 77, False), (128, 2049, False), (16, 300, False),
                                     (128, 2049, True), (32, 5, True)])
def test_decode_bounds_checked(libs, d, n0, vt):
    normal, checked = libs
    B_, H, T = 1, 3, 3
    kc, vc = inputs.make_decode_cache(B_, H, n0, d, n0 + T, "bf16", seed=5)
    steps = [t.cuda() for t in inputs.make_decode_steps(B_, H, d, T, "bf16", seed=5)]

    def run():
        k, v = kc.cuda(), vc.cuda()
        ws = P.alloc_workspace(P.path_decode_workspace_bytes(B_, H, n0 + T, d), "cuda")
        outs = []
        for t in range(T):
            outs.append(P.path_decode_step(*(s[t] for s in steps), k, v, n0 + t, workspace=ws, value_transport=vt))
        torch.cuda.synchronize()
        return torch.stack(outs), k, v, P.path_get_status(ws)

    o1, k1, v1, st1 = _with(normal, run)
    o2, k2, v2, st2 = _with(checked, run)
    assert st1 == P.PATH_OK and st2 == P.PATH_OK, (st1, st2)
    assert torch.equal(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)
