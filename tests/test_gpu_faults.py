"""Device-side failure path (GPU), without a fault: the test hook makes the TMA producer of the
tensor-core forward skip one signal, so the MMA warp's bounded wait (20 ms under the hook)
expires.  The kernel must record PATH_ERR_TIMEOUT in the workspace status word, drain, free
TMEM and return; the context stays usable and the next call is correct again."""
import numpy as np
import pytest
import torch

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import inputs
from gpu_common import check, to_np
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    x = inputs.make_fwd(1, 2, 384, 128, "bf16", seed=41)  # three query tiles: the hook hits the scan
    args = [t.cuda() for t in (x.q, x.k, x.v, x.w, x.beta)]
    ws = P.alloc_workspace(P.path_attn_workspace_bytes(1, 2, 384, 128, torch.bfloat16), "cuda")
    try:
        P.path_debug_set_fault(1)
        P.path_attn_fwd(*args, scale=x.scale, workspace=ws)
        assert P.path_get_status(ws) == P.PATH_ERR_TIMEOUT
    finally:
        P.path_debug_set_fault(0)
    o = P.path_attn_fwd(*args, scale=x.scale, workspace=ws)
    assert P.path_get_status(ws) == P.PATH_OK
    f = inputs.f64
    ref, _ = orc.path_attn(f(x.q), f(x.k), f(x.v), f(x.w), f(x.beta), None, x.scale)
    check(to_np(o), ref, torch.bfloat16, "after timeout")
