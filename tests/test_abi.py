"""C-ABI library: loads, exports every symbol include/path_attn.h declares, and rejects bad
arguments synchronously before any launch (CPU only: no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

import attention_causal_attn_fwd_gb300 as P
from attention_causal_attn_fwd_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(P.LIB_PATH):
        B.build()
    return P.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "path_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(path_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "path_attn_fwd" in names and "path_decode_step" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(P.EXPORTED)


def test_status_strings_and_version(lib):
    assert lib.path_version() >= 1
    for code in range(6):
        assert P.status_string(code)
    assert P.status_string(P.PATH_ERR_TIMEOUT) == "device-side wait timed out"


def test_workspace_sizes(lib):
    import torch
    assert P.path_attn_workspace_bytes(8, 12, 4096, 128, torch.bfloat16) > 8 * 12 * 4096 * 128 * 4
    assert P.path_attn_workspace_bytes(1, 1, 64, 16, torch.float32) > 0
    assert P.path_attn_workspace_bytes(1, 1, 64, 48, torch.float32) == 0      # unsupported d
    assert P.path_attn_workspace_bytes(1, 1, 64, 16, torch.bfloat16) == 0     # bf16 tensor-core path: d in {64,128}
    assert P.path_decode_workspace_bytes(64, 12, 33024, 128) > 0
    assert P.path_decode_workspace_bytes(1, 1, 10, 48) == 0


FAKE = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never dereferenced: calls below fail validation first


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, w=FAKE, beta=FAKE, o=FAKE, lse=None, B=1, H=1, L=64, d=16, dt=P.PATH_F32,
             causal=1, scale=ctypes.c_float(0.25), ws=FAKE, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.path_attn_fwd(a["q"], a["k"], a["v"], a["w"], a["beta"], a["o"], a["lse"], a["B"], a["H"], a["L"],
                             a["d"], a["dt"], a["causal"], a["scale"], a["ws"], a["ws_bytes"], a["stream"])


def test_forward_argument_errors(lib):
    assert _fwd(lib, causal=0) == P.PATH_ERR_UNSUPPORTED
    assert _fwd(lib, d=48) == P.PATH_ERR_UNSUPPORTED
    assert _fwd(lib, dt=7) == P.PATH_ERR_UNSUPPORTED
    assert _fwd(lib, L=0) == P.PATH_ERR_INVALID
    assert _fwd(lib, B=-1) == P.PATH_ERR_INVALID
    assert _fwd(lib, q=None) == P.PATH_ERR_INVALID
    assert _fwd(lib, v=ctypes.c_void_p((1 << 20) + 4)) == P.PATH_ERR_INVALID  # misaligned
    assert _fwd(lib, ws_bytes=16) == P.PATH_ERR_WORKSPACE
    assert _fwd(lib, ws=None, ws_bytes=1 << 30) == P.PATH_ERR_WORKSPACE
    assert _fwd(lib, B=300, H=300, L=1) == P.PATH_ERR_UNSUPPORTED  # B*H above the grid limit (65535)
    fox = lib.path_attn_fwd_fox(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 1, 64, 16, P.PATH_F32, 1,
                                ctypes.c_float(0.25), FAKE, 1 << 30, None)
    assert fox == P.PATH_ERR_INVALID  # log_f is required
    rel = lib.path_attn_fwd_relbias(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 1, 64, 16, P.PATH_F32, 1,
                                    ctypes.c_float(0.25), FAKE, 1 << 30, None)
    assert rel == P.PATH_ERR_INVALID  # rel_bias is required
    rel = lib.path_attn_fwd_relbias(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_void_p((1 << 20) + 8), FAKE, None, 1, 1,
                                    64, 16, P.PATH_F32, 1, ctypes.c_float(0.25), FAKE, 1 << 30, None)
    assert rel == P.PATH_ERR_INVALID  # misaligned table
    rel = lib.path_attn_fwd_relbias(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 1, 64, 16, P.PATH_F32, 0,
                                    ctypes.c_float(0.25), FAKE, 1 << 30, None)
    assert rel == P.PATH_ERR_UNSUPPORTED  # non-causal


def test_bwd_argument_errors(lib):
    def bwd(**kw):
        a = dict(log_f=None, dlog_f=None, lse=FAKE, d=64, dt=P.PATH_BF16, causal=1, BH=(2, 3), L=300,
                 ws_bytes=1 << 40, dq=FAKE)
        a.update(kw)
        B, H = a["BH"]
        return lib.path_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, a["log_f"], FAKE, a["lse"], FAKE, a["dq"], FAKE, FAKE,
                                 FAKE, FAKE, a["dlog_f"], B, H, a["L"], a["d"], a["dt"], a["causal"],
                                 ctypes.c_float(0.125), FAKE, a["ws_bytes"], None)
    assert bwd(L=0) == P.PATH_ERR_INVALID                 # empty sequence
    assert bwd(BH=(0, 3)) == P.PATH_ERR_INVALID
    assert bwd(lse=None) == P.PATH_ERR_INVALID            # the forward's lse is required
    assert bwd(dq=None) == P.PATH_ERR_INVALID
    assert bwd(log_f=FAKE) == P.PATH_ERR_INVALID          # FoX needs dlog_f
    assert bwd(dq=ctypes.c_void_p((1 << 20) + 4)) == P.PATH_ERR_INVALID  # misaligned
    assert bwd(d=48) == P.PATH_ERR_UNSUPPORTED
    assert bwd(dt=7) == P.PATH_ERR_UNSUPPORTED
    assert bwd(causal=0) == P.PATH_ERR_UNSUPPORTED
    assert bwd(BH=(300, 300)) == P.PATH_ERR_UNSUPPORTED   # B*H above the grid limit
    assert bwd(ws_bytes=4096) == P.PATH_ERR_WORKSPACE
    need = lib.path_attn_bwd_workspace_bytes(2, 3, 300, 64, P.PATH_BF16)
    # 5 chunks of 64: 10 (query chunk, key chunk) pairs per head hold U, G (64 x 64), dS and P (64 x 64),
    # in the input dtype (bf16 here; fp32 pairs for fp32 inputs)
    assert need > 6 * 10 * (2 * 64 * 64 + 2 * 64 * 64) * 2
    need32 = lib.path_attn_bwd_workspace_bytes(2, 3, 300, 64, P.PATH_F32)
    assert need32 - need >= 6 * 10 * (2 * 64 * 64 + 2 * 64 * 64) * 2
    assert lib.path_attn_bwd_workspace_bytes(2, 3, 300, 48, P.PATH_BF16) == 0
    assert lib.path_attn_bwd_workspace_bytes(2, 3, 300, 64, 9) == 0


def test_decode_argument_errors(lib):
    def step(**kw):
        a = dict(n_cached=10, n_max=11, d=128, dt=P.PATH_BF16, ws_bytes=1 << 30, kc=FAKE)
        a.update(kw)
        return lib.path_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, a["kc"], FAKE, a["n_cached"], a["n_max"], FAKE,
                                    None, 2, 3, a["d"], ctypes.c_float(0.1), a["dt"], FAKE, a["ws_bytes"], None)
    assert step(n_cached=11, n_max=11) == P.PATH_ERR_INVALID  # no room for the new token
    assert step(n_cached=-1) == P.PATH_ERR_INVALID
    assert step(d=48) == P.PATH_ERR_UNSUPPORTED
    assert step(dt=3) == P.PATH_ERR_UNSUPPORTED
    assert step(kc=None) == P.PATH_ERR_INVALID
    assert step(ws_bytes=8) == P.PATH_ERR_WORKSPACE
    assert lib.path_kcache_update(FAKE, 2, 3, 12, 11, 128, FAKE, FAKE, P.PATH_BF16, None) == P.PATH_ERR_INVALID
    assert lib.path_kcache_update(FAKE, 2, 3, 5, 11, 100, FAKE, FAKE, P.PATH_BF16, None) == P.PATH_ERR_UNSUPPORTED
    # B*H goes on a grid dimension limited to 65535: rejected before any launch (d = 16 with a short cache
    # would otherwise fit the no-alloc scratch too)
    big = lib.path_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, FAKE, None, 256, 257, 16,
                               ctypes.c_float(0.25), P.PATH_BF16, FAKE, 1 << 40, None)
    assert big == P.PATH_ERR_UNSUPPORTED
    assert lib.path_kcache_update(FAKE, 256, 257, 1, 2, 16, FAKE, FAKE, P.PATH_BF16, None) == P.PATH_ERR_UNSUPPORTED
    assert lib.path_decode_step_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, FAKE, None, 256, 257, 16,
                                        ctypes.c_float(0.25), P.PATH_BF16, None) == P.PATH_ERR_UNSUPPORTED
    assert lib.path_prefill_kcache(FAKE, FAKE, FAKE, FAKE, 256, 257, 1, 1, 128, P.PATH_BF16, FAKE, 1 << 40,
                                   None) == P.PATH_ERR_UNSUPPORTED


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 1, 8, 16)
    with pytest.raises(ValueError):
        P.path_attn_fwd(x, x, x, x, torch.zeros(1, 1, 8))


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(P.PathLibraryError):
        P.load(str(tmp_path / "nope.so"))


def test_package_does_not_import_the_oracle():
    """The product path never reaches oracle/ (no import, no call)."""
    pkg = os.path.join(ROOT, "attention_causal_attn_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"(import\s+oracle|from\s+oracle|oracle/|path_oracle)", src), f


def test_noalloc_decode_rejects_sizes_beyond_its_scratch(lib):
    """The allocation-free decode step refuses, before touching the GPU, any size whose
    scratch would not fit in its built-in PATH_DECODE_NOALLOC_SCRATCH_BYTES (8 MiB)."""
    limit = 8 << 20
    assert P.path_decode_workspace_bytes(64, 12, 43008, 128) <= limit
    assert P.path_decode_workspace_bytes(64, 12, 65537, 128) > limit
    rc = lib.path_decode_step_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 65536, 65537, FAKE, None, 64, 12,
                                      128, ctypes.c_float(0.1), P.PATH_BF16, None)
    assert rc == P.PATH_ERR_WORKSPACE
    assert lib.path_decode_step_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 5, 5, FAKE, None, 1, 1, 128,
                                        ctypes.c_float(0.1), P.PATH_BF16, None) == P.PATH_ERR_INVALID


def test_prefill_argument_errors(lib):
    def call(**kw):
        a = dict(L=100, n_max=100, d=128, dt=P.PATH_BF16, ws_bytes=1 << 34, kc=FAKE)
        a.update(kw)
        return lib.path_prefill_kcache(FAKE, FAKE, FAKE, a["kc"], 1, 2, a["L"], a["n_max"], a["d"], a["dt"], FAKE,
                                       a["ws_bytes"], None)
    assert call(n_max=99) == P.PATH_ERR_INVALID      # the cache cannot hold the prompt
    assert call(L=0) == P.PATH_ERR_INVALID
    assert call(d=16) == P.PATH_ERR_UNSUPPORTED       # bf16 path: d in {64, 128}
    assert call(kc=None) == P.PATH_ERR_INVALID
    assert call(ws_bytes=64) == P.PATH_ERR_WORKSPACE
    assert lib.path_prefill_workspace_bytes(1, 2, 100, 128, P.PATH_BF16) > lib.path_attn_workspace_bytes(
        1, 2, 100, 128, P.PATH_BF16)
