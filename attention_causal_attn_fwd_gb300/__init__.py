"""PaTH causal attention (forward, PaTH-FoX forward, decode) on GB300 (sm_103a).

Thin ctypes binding over libpathattn.so (C ABI in include/path_attn.h).  Every
step of the computation runs in the library's CUDA kernels; this module only
checks tensor layouts, allocates outputs and workspaces through torch, and
passes raw device pointers plus the current CUDA stream.  There is no CPU
fallback: a missing library raises ``PathLibraryError``.

Functions keep the C names:

- ``path_attn_fwd(q, k, v, w, beta, scale=None, lse=False)``
- ``path_attn_fwd_fox(q, k, v, w, beta, log_f, scale=None, lse=False)``
- ``path_attn_fwd_relbias(q, k, v, w, beta, rel_bias, scale=None, lse=False)``
- ``path_decode_step(q_t, k_t, v_t, w_t, beta_t, kcache, vcache, n_cached, scale=None, value_transport=False)``
- ``path_attn_fwd_vt(q, k, v, w, beta, log_f=None, scale=None, lse=False)`` (value-side transport)
- ``path_kcache_update(kcache, n_cached, w_t, beta_t)``
- ``path_get_status(workspace)``, ``path_fwd_visited_blocks(workspace)``, ``path_attn_workspace_bytes(...)``,
  ``path_decode_workspace_bytes(...)``
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpathattn.so")

(PATH_OK, PATH_ERR_INVALID, PATH_ERR_UNSUPPORTED, PATH_ERR_CUDA, PATH_ERR_TIMEOUT, PATH_ERR_WORKSPACE,
 PATH_ERR_BOUNDS) = range(7)
PATH_F32, PATH_BF16 = 0, 1
_DT = {torch.float32: PATH_F32, torch.bfloat16: PATH_BF16}

EXPORTED = ("path_version", "path_status_string", "path_attn_workspace_bytes", "path_attn_fwd",
            "path_attn_fwd_fox", "path_decode_workspace_bytes", "path_kcache_update", "path_decode_step",
            "path_get_status", "path_debug_set_fault", "path_debug_set_timing_events", "path_decode_step_noalloc",
            "path_prefill_workspace_bytes", "path_prefill_kcache", "path_attn_fwd_relbias",
            "path_attn_bwd_workspace_bytes", "path_attn_bwd", "path_fwd_visited_blocks", "path_debug_set_fox_skip",
            "path_decode_step_vt", "path_attn_fwd_vt_workspace_bytes", "path_attn_fwd_vt")


class PathLibraryError(RuntimeError):
    """libpathattn.so is missing or could not be loaded."""


class PathError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (status %d)" % (where, status_string(code), code))


_lib = None
_vp, _fp, _i, _sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpathattn.so (build it with ``attention_causal_attn_fwd_gb300.build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise PathLibraryError("libpathattn.so not found at %s; run __graft_entry__.build()" % p)
    try:
        lib = ctypes.CDLL(p)
    except OSError as e:
        raise PathLibraryError("cannot load %s: %s" % (p, e)) from e
    lib.path_version.restype = _i
    lib.path_status_string.argtypes = [_i]
    lib.path_status_string.restype = ctypes.c_char_p
    lib.path_attn_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
    lib.path_attn_workspace_bytes.restype = _sz
    lib.path_attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _fp, _vp, _fp, _i, _i, _i, _i, _i, _i, ctypes.c_float, _vp,
                                  _sz, _vp]
    lib.path_attn_fwd.restype = _i
    lib.path_attn_fwd_fox.argtypes = [_vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp, _i, _i, _i, _i, _i, _i,
                                      ctypes.c_float, _vp, _sz, _vp]
    lib.path_attn_fwd_fox.restype = _i
    lib.path_attn_fwd_relbias.argtypes = lib.path_attn_fwd_fox.argtypes
    lib.path_attn_fwd_relbias.restype = _i
    lib.path_attn_bwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
    lib.path_attn_bwd_workspace_bytes.restype = _sz
    lib.path_attn_bwd.argtypes = [_vp, _vp, _vp, _vp, _fp, _fp, _vp, _fp, _vp, _vp, _vp, _vp, _vp, _fp, _fp,
                                  _i, _i, _i, _i, _i, _i, ctypes.c_float, _vp, _sz, _vp]
    lib.path_attn_bwd.restype = _i
    lib.path_decode_workspace_bytes.argtypes = [_i, _i, _i, _i]
    lib.path_decode_workspace_bytes.restype = _sz
    lib.path_kcache_update.argtypes = [_vp, _i, _i, _i, _i, _i, _vp, _fp, _i, _vp]
    lib.path_kcache_update.restype = _i
    lib.path_decode_step.argtypes = [_vp, _vp, _vp, _vp, _fp, _vp, _vp, _i, _i, _vp, _fp, _i, _i, _i,
                                     ctypes.c_float, _i, _vp, _sz, _vp]
    lib.path_decode_step.restype = _i
    lib.path_decode_step_vt.argtypes = lib.path_decode_step.argtypes
    lib.path_decode_step_vt.restype = _i
    lib.path_attn_fwd_vt_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
    lib.path_attn_fwd_vt_workspace_bytes.restype = _sz
    lib.path_attn_fwd_vt.argtypes = lib.path_attn_fwd_fox.argtypes
    lib.path_attn_fwd_vt.restype = _i
    lib.path_decode_step_noalloc.argtypes = [_vp, _vp, _vp, _vp, _fp, _vp, _vp, _i, _i, _vp, _fp, _i, _i, _i,
                                             ctypes.c_float, _i, _vp]
    lib.path_decode_step_noalloc.restype = _i
    lib.path_prefill_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
    lib.path_prefill_workspace_bytes.restype = _sz
    lib.path_prefill_kcache.argtypes = [_vp, _vp, _fp, _vp, _i, _i, _i, _i, _i, _i, _vp, _sz, _vp]
    lib.path_prefill_kcache.restype = _i
    lib.path_get_status.argtypes = [_vp, _vp]
    lib.path_get_status.restype = _i
    lib.path_debug_set_fault.argtypes = [_i]
    lib.path_debug_set_fault.restype = None
    lib.path_debug_set_timing_events.argtypes = [_vp, _vp]
    lib.path_debug_set_timing_events.restype = None
    lib.path_fwd_visited_blocks.argtypes = [_vp, _vp]
    lib.path_fwd_visited_blocks.restype = ctypes.c_longlong
    lib.path_debug_set_fox_skip.argtypes = [_i]
    lib.path_debug_set_fox_skip.restype = None
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().path_status_string(int(code)).decode()
    except PathLibraryError:
        return "status %d" % code


def _check(code: int, where: str):
    if code != PATH_OK:
        raise PathError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


def path_attn_workspace_bytes(B: int, H: int, L: int, d: int, dtype: torch.dtype) -> int:
    return int(load().path_attn_workspace_bytes(B, H, L, d, _DT[dtype]))


def path_decode_workspace_bytes(B: int, H: int, n_max: int, d: int) -> int:
    return int(load().path_decode_workspace_bytes(B, H, n_max, d))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """A device workspace buffer of at least nbytes (uint8, 256-byte aligned by torch)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _fwd(q, k, v, w, beta, log_f, scale, lse, out, ws, rel_bias=None):
    lib = load()
    if q.dim() != 4:
        raise ValueError("q must be [B, H, L, d]")
    B, H, L, d = q.shape
    dt = q.dtype
    if dt not in _DT:
        raise ValueError("dtype must be float32 or bfloat16")
    for name, t in (("q", q), ("k", k), ("v", v), ("w", w)):
        _dev(t, name, dt, (B, H, L, d))
    _dev(beta, "beta", torch.float32, (B, H, L))
    if log_f is not None:
        _dev(log_f, "log_f", torch.float32, (B, H, L))
    if rel_bias is not None:
        _dev(rel_bias, "rel_bias", torch.float32, (H, L))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else _dev(out, "out", dt, (B, H, L, d))
    lse_t = torch.empty((B, H, L), dtype=torch.float32, device=q.device) if lse else None
    need = lib.path_attn_workspace_bytes(B, H, L, d, _DT[dt])
    if need == 0:
        raise PathError(PATH_ERR_UNSUPPORTED, "path_attn_fwd")
    if ws is None:
        ws = alloc_workspace(need, q.device)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta)]
    tail = [_ptr(o), _ptr(lse_t), B, H, L, d, _DT[dt], 1, ctypes.c_float(scale), _ptr(ws), ws.numel(), _stream()]
    if rel_bias is not None:
        _check(lib.path_attn_fwd_relbias(*args, _ptr(rel_bias), *tail), "path_attn_fwd_relbias")
    elif log_f is None:
        _check(lib.path_attn_fwd(*args, *tail), "path_attn_fwd")
    else:
        _check(lib.path_attn_fwd_fox(*args, _ptr(log_f), *tail), "path_attn_fwd_fox")
    return (o, lse_t) if lse else o


def path_attn_fwd(q, k, v, w, beta, scale=None, lse=False, out=None, workspace=None):
    """PaTH causal attention forward.  q, k, v, w: [B, H, L, d] CUDA (fp32 or bf16); beta [B, H, L] fp32."""
    return _fwd(q, k, v, w, beta, None, scale, lse, out, workspace)


def path_attn_fwd_fox(q, k, v, w, beta, log_f, scale=None, lse=False, out=None, workspace=None):
    """PaTH-FoX forward: adds sum_{s=j+1..i} log_f[s] to the scaled logit of (i, j)."""
    if log_f is None:
        raise ValueError("log_f is required")
    return _fwd(q, k, v, w, beta, log_f, scale, lse, out, workspace)


def path_attn_fwd_relbias(q, k, v, w, beta, rel_bias, scale=None, lse=False, out=None, workspace=None):
    """PaTH forward with a relative-position bias: adds rel_bias[h, i - j] to the scaled logit of (i, j).

    rel_bias: [H, L] fp32 CUDA, shared by every batch entry (e.g. a GGD-BAM or ALiBi prior)."""
    if rel_bias is None:
        raise ValueError("rel_bias is required")
    return _fwd(q, k, v, w, beta, None, scale, lse, out, workspace, rel_bias=rel_bias)


def path_attn_fwd_vt(q, k, v, w, beta, log_f=None, scale=None, lse=False, out=None, workspace=None):
    """PaTH(-FoX) forward with value-side transport: o_i = sum_j softmax_j(s_i.) H_i ... H_{j+1} v_j."""
    lib = load()
    if q.dim() != 4:
        raise ValueError("q must be [B, H, L, d]")
    B, H, L, d = q.shape
    dt = q.dtype
    if dt not in _DT:
        raise ValueError("dtype must be float32 or bfloat16")
    for name, t in (("q", q), ("k", k), ("v", v), ("w", w)):
        _dev(t, name, dt, (B, H, L, d))
    _dev(beta, "beta", torch.float32, (B, H, L))
    if log_f is not None:
        _dev(log_f, "log_f", torch.float32, (B, H, L))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else _dev(out, "out", dt, (B, H, L, d))
    lse_t = torch.empty((B, H, L), dtype=torch.float32, device=q.device) if lse else None
    need = lib.path_attn_fwd_vt_workspace_bytes(B, H, L, d, _DT[dt])
    if need == 0:
        raise PathError(PATH_ERR_UNSUPPORTED, "path_attn_fwd_vt")
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    _check(lib.path_attn_fwd_vt(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(log_f), _ptr(o), _ptr(lse_t),
                                B, H, L, d, _DT[dt], 1, ctypes.c_float(scale), _ptr(workspace), workspace.numel(),
                                _stream()), "path_attn_fwd_vt")
    return (o, lse_t) if lse else o


def path_attn_bwd_workspace_bytes(B: int, H: int, L: int, d: int, dtype: torch.dtype) -> int:
    return int(load().path_attn_bwd_workspace_bytes(B, H, L, d, _DT[dtype]))


def path_attn_bwd(q, k, v, w, beta, o, lse, dO, log_f=None, scale=None, workspace=None):
    """Gradients of PaTH (or, with log_f, PaTH-FoX) attention for a loss with gradient dO w.r.t. o.

    q, k, v, w, dO and the forward output o: [B, H, L, d] CUDA (fp32 or bf16); beta, lse (the
    forward's log-sum-exp) and log_f: [B, H, L] fp32.  Returns a dict with dq, dk, dv, dw (dtype of
    q), dbeta and, with log_f, dlog_f (fp32)."""
    lib = load()
    if q.dim() != 4:
        raise ValueError("q must be [B, H, L, d]")
    B, H, L, d = q.shape
    dt = q.dtype
    if dt not in _DT:
        raise ValueError("dtype must be float32 or bfloat16")
    for name, t in (("q", q), ("k", k), ("v", v), ("w", w), ("o", o), ("dO", dO)):
        _dev(t, name, dt, (B, H, L, d))
    for name, t in (("beta", beta), ("lse", lse)) + ((("log_f", log_f),) if log_f is not None else ()):
        _dev(t, name, torch.float32, (B, H, L))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = {n: torch.empty_like(q) for n in ("dq", "dk", "dv", "dw")}
    out["dbeta"] = torch.empty_like(beta)
    if log_f is not None:
        out["dlog_f"] = torch.empty_like(beta)
    need = lib.path_attn_bwd_workspace_bytes(B, H, L, d, _DT[dt])
    if need == 0:
        raise PathError(PATH_ERR_UNSUPPORTED, "path_attn_bwd")
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    _check(lib.path_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(log_f), _ptr(o), _ptr(lse),
                             _ptr(dO), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dw"]),
                             _ptr(out["dbeta"]), _ptr(out.get("dlog_f")), B, H, L, d, _DT[dt], 1,
                             ctypes.c_float(scale), _ptr(workspace), workspace.numel(), _stream()),
           "path_attn_bwd")
    return out


def path_prefill_workspace_bytes(B: int, H: int, L: int, d: int, dtype: torch.dtype) -> int:
    return int(load().path_prefill_workspace_bytes(B, H, L, d, _DT[dtype]))


def path_prefill_kcache(k, w, beta, kcache=None, n_max=None, workspace=None):
    """Transported key cache of a prompt: kcache[:, :, j] = H_{L-1} ... H_{j+1} k[:, :, j] for j < L.

    k, w: [B, H, L, d] CUDA (fp32 or bf16); beta [B, H, L] fp32.  Allocates kcache [B, H, n_max, d]
    (n_max defaults to L) unless one is given; returns it.  Decoding continues with n_cached = L.
    """
    lib = load()
    B, H, L, d = k.shape
    dt = k.dtype
    _dev(k, "k", dt, (B, H, L, d))
    _dev(w, "w", dt, (B, H, L, d))
    _dev(beta, "beta", torch.float32, (B, H, L))
    if kcache is None:
        kcache = torch.zeros((B, H, n_max or L, d), dtype=dt, device=k.device)
    _dev(kcache, "kcache", dt)
    need = lib.path_prefill_workspace_bytes(B, H, L, d, _DT[dt])
    if need == 0:
        raise PathError(PATH_ERR_UNSUPPORTED, "path_prefill_kcache")
    ws = alloc_workspace(need, k.device) if workspace is None else workspace
    _check(lib.path_prefill_kcache(_ptr(k), _ptr(w), _ptr(beta), _ptr(kcache), B, H, L, kcache.shape[2], d,
                                   _DT[dt], _ptr(ws), ws.numel(), _stream()), "path_prefill_kcache")
    return kcache


def path_kcache_update(kcache, n_cached: int, w_t, beta_t):
    """In place: kcache[:, :, j] <- (I - beta_t w_t w_t^T) kcache[:, :, j] for j < n_cached."""
    lib = load()
    B, H, n_max, d = kcache.shape
    _dev(kcache, "kcache")
    _dev(w_t, "w_t", kcache.dtype, (B, H, d))
    _dev(beta_t, "beta_t", torch.float32, (B, H))
    _check(lib.path_kcache_update(_ptr(kcache), B, H, int(n_cached), n_max, d, _ptr(w_t), _ptr(beta_t),
                                  _DT[kcache.dtype], _stream()), "path_kcache_update")


def path_decode_step(q_t, k_t, v_t, w_t, beta_t, kcache, vcache, n_cached: int, scale=None, out=None,
                     lse=False, workspace=None, value_transport=False):
    """One decode step for all heads; updates kcache/vcache in place and returns o_t [B, H, d].

    value_transport=True calls path_decode_step_vt: the value cache is transported in place with the keys."""
    lib = load()
    B, H, n_max, d = kcache.shape
    dt = kcache.dtype
    _dev(kcache, "kcache")
    _dev(vcache, "vcache", dt, (B, H, n_max, d))
    for name, t in (("q_t", q_t), ("k_t", k_t), ("v_t", v_t), ("w_t", w_t)):
        _dev(t, name, dt, (B, H, d))
    _dev(beta_t, "beta_t", torch.float32, (B, H))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q_t) if out is None else out
    lse_t = torch.empty((B, H), dtype=torch.float32, device=q_t.device) if lse else None
    if workspace is None:
        workspace = alloc_workspace(lib.path_decode_workspace_bytes(B, H, n_max, d), q_t.device)
    fn, name = (lib.path_decode_step_vt, "path_decode_step_vt") if value_transport else \
        (lib.path_decode_step, "path_decode_step")
    _check(fn(_ptr(q_t), _ptr(k_t), _ptr(v_t), _ptr(w_t), _ptr(beta_t), _ptr(kcache), _ptr(vcache), int(n_cached),
              n_max, _ptr(o), _ptr(lse_t), B, H, d, ctypes.c_float(scale), _DT[dt], _ptr(workspace),
              workspace.numel(), _stream()), name)
    return (o, lse_t) if lse else o


def path_get_status(workspace_tensor) -> int:
    """Status word of the last call that used this workspace (synchronises the current stream)."""
    return int(load().path_get_status(_ptr(workspace_tensor), _stream()))


def path_fwd_visited_blocks(workspace_tensor) -> int:
    """(query tile, key block) pairs the last bf16 forward on this workspace visited (synchronises)."""
    return int(load().path_fwd_visited_blocks(_ptr(workspace_tensor), _stream()))


def path_debug_set_fox_skip(enabled: bool):
    """Turn the PaTH-FoX far-block stop of the bf16 forward on (default) or off (visit every block)."""
    load().path_debug_set_fox_skip(1 if enabled else 0)


def path_debug_set_fault(mask: int):
    load().path_debug_set_fault(int(mask))


def path_debug_set_timing_events(ev_start=None, ev_end=None):
    """Record two torch.cuda.Events around the dominant kernel of each later call (None, None stops)."""
    h = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)
    load().path_debug_set_timing_events(h(ev_start), h(ev_end))


def path_decode_step_noalloc(q_t, k_t, v_t, w_t, beta_t, kcache, vcache, n_cached: int, scale=None, out=None,
                             lse=False):
    """path_decode_step without a workspace: for callers that cannot allocate device memory while decoding.

    The library's built-in scratch (PATH_DECODE_NOALLOC_SCRATCH_BYTES = 8 MiB per GPU) replaces the
    workspace; sizes that need more raise PathError(PATH_ERR_WORKSPACE).  Calls that may overlap on the
    GPU share that scratch and must be ordered.  Pass ``out`` (and no ``lse``) to avoid any allocation
    here as well.
    """
    lib = load()
    B, H, n_max, d = kcache.shape
    dt = kcache.dtype
    _dev(kcache, "kcache")
    _dev(vcache, "vcache", dt, (B, H, n_max, d))
    for name, t in (("q_t", q_t), ("k_t", k_t), ("v_t", v_t), ("w_t", w_t)):
        _dev(t, name, dt, (B, H, d))
    _dev(beta_t, "beta_t", torch.float32, (B, H))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q_t) if out is None else out
    lse_t = torch.empty((B, H), dtype=torch.float32, device=q_t.device) if lse else None
    _check(lib.path_decode_step_noalloc(_ptr(q_t), _ptr(k_t), _ptr(v_t), _ptr(w_t), _ptr(beta_t), _ptr(kcache),
                                        _ptr(vcache), int(n_cached), n_max, _ptr(o), _ptr(lse_t), B, H, d,
                                        ctypes.c_float(scale), _DT[dt], _stream()), "path_decode_step_noalloc")
    return (o, lse_t) if lse else o
