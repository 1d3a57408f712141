"""fp64 CPU oracle for PaTH causal attention (ctypes wrapper) — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
``--impl reference`` leg may import this module.  It never imports the CUDA
package and the CUDA package never imports it.

The arithmetic lives in ``oracle/path_oracle.c``: a plain backward walk of each
query through the transitions H_s = I - beta_s w_s w_s^T, in fp64, following
"Resumo Técnico: Atenção PaTH" (gist.science/pt/paper/2505.16381), §2
"Mecanismo Central" (logit and transition equations), §2 "Extensões: PaTH-FoX"
(additive forget-gate bias) and §3 "Inferência" (in-place key update).

Pins: tests/test_oracle.py checks this oracle against an explicit dense product
of d x d matrices (brute force), against library causal attention at beta = 0,
closed forms (d = 1; constant w with beta = 2), orthogonality at beta = 2,
decode = prefill, and hand-derived golden logits (tests/golden/).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "path_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpath_oracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math).  Returns the .so path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.path_oracle_fwd_rows.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_double, _i64p, ctypes.c_int64, _dp, _dp]
            lib.path_oracle_fwd_rows.restype = None
            lib.path_oracle_fwd_rows_relbias.argtypes = lib.path_oracle_fwd_rows.argtypes
            lib.path_oracle_fwd_rows_relbias.restype = None
            lib.path_oracle_fwd_rows_vt.argtypes = lib.path_oracle_fwd_rows.argtypes
            lib.path_oracle_fwd_rows_vt.restype = None
            lib.path_oracle_logits.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double, _dp]
            lib.path_oracle_logits.restype = None
            lib.path_oracle_decode.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp,
                                               _dp, _dp, _dp, ctypes.c_int, ctypes.c_double, _dp, _dp]
            lib.path_oracle_decode.restype = None
            lib.path_oracle_decode_vt.argtypes = lib.path_oracle_decode.argtypes
            lib.path_oracle_decode_vt.restype = None
            lib.path_oracle_kcache_update.argtypes = [_dp, ctypes.c_int, ctypes.c_int, _dp, ctypes.c_double]
            lib.path_oracle_kcache_update.restype = None
            lib.path_oracle_bwd.argtypes = [_dp] * 7 + [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_double] + [_dp] * 6
            lib.path_oracle_bwd.restype = None
            lib.path_oracle_threads.argtypes = []
            lib.path_oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses (honours OMP_NUM_THREADS)."""
    return int(_load().path_oracle_threads())


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def path_attn(q, k, v, w, beta, log_f=None, scale=None, rows=None, rel_bias=None, value_transport=False):
    """Causal PaTH(-FoX) attention in fp64.

    q, k, v, w: [..., L, d]; beta, log_f: [..., L].  Leading dims are flattened
    into heads.  ``rows`` (optional, int array) selects flat row indices
    ``head * L + i``; then o is [len(rows), d] and lse [len(rows)].  Otherwise
    o has q's shape and lse q's shape without d.

    ``rel_bias`` ([..., L] like beta; exclusive with log_f) adds rel_bias[..., i - j]
    unscaled to the logit of (i, j): a relative-position prior such as GGD-BAM's
    ("Resumo Técnico: Mecanismo de Atenção Bayesiana (BAM)", §"Solução Proposta:
    GGD-BAM") or ALiBi's, on top of the PaTH logits.

    ``value_transport`` (exclusive with rel_bias) carries every value along the route to its query:
    o_i = sum_j alpha_ij H_i ... H_{j+1} v_j ("Resumo Técnico: Por que Transformações Acumuladas
    Extrapolam?", §"Principais Contribuições" 3 "Proteção do Lado de Valor").
    """
    q, k, v, w, beta = (_f64(x) for x in (q, k, v, w, beta))
    lf = None if log_f is None else _f64(log_f)
    rb = None if rel_bias is None else _f64(rel_bias)
    assert lf is None or rb is None, "log_f and rel_bias are exclusive"
    L, d = q.shape[-2], q.shape[-1]
    BH = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    for x in (k, v, w):
        assert x.shape == q.shape
    assert beta.shape == q.shape[:-1]
    if lf is not None:
        assert lf.shape == beta.shape
    if rb is not None:
        assert rb.shape == beta.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    lib = _load()
    assert not (value_transport and rb is not None), "value transport takes no relative bias"
    fn, extra = (lib.path_oracle_fwd_rows, lf) if rb is None else (lib.path_oracle_fwd_rows_relbias, rb)
    if value_transport:
        fn = lib.path_oracle_fwd_rows_vt
    if rows is None:
        n = BH * L
        o = np.empty((n, d))
        lse = np.empty(n)
        fn(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(extra), BH, L, d, float(scale), None, n,
           _ptr(o), _ptr(lse))
        return o.reshape(q.shape), lse.reshape(q.shape[:-1])
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rows.min() >= 0 and rows.max() < BH * L
    o = np.empty((rows.size, d))
    lse = np.empty(rows.size)
    fn(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(extra), BH, L, d, float(scale),
       rows.ctypes.data_as(_i64p), rows.size, _ptr(o), _ptr(lse))
    return o, lse


def path_logits(q, k, w, beta, log_f=None, scale=1.0):
    """Full [L, L] logit matrix of one head (j > i set to -inf); tiny inputs only."""
    q, k, w, beta = (_f64(x) for x in (q, k, w, beta))
    lf = None if log_f is None else _f64(log_f)
    L, d = q.shape
    S = np.empty((L, L))
    _load().path_oracle_logits(_ptr(q), _ptr(k), _ptr(w), _ptr(beta), _ptr(lf), L, d, float(scale), _ptr(S))
    return S


def path_decode(kc0, vc0, q, k, v, w, beta, scale, value_transport=False):
    """Decode T steps of ONE head from a cache of n0 transported keys.

    kc0, vc0: [n0, d]; q, k, v, w: [T, d]; beta: [T].  Returns (o [T, d],
    lse [T], kc [n0+T, d], vc [n0+T, d]) where kc holds the final transported keys
    (and, with ``value_transport``, vc the transported values, vc0 being values
    already carried to the cache's position).
    """
    kc0, vc0, q, k, v, w, beta = (_f64(x) for x in (kc0, vc0, q, k, v, w, beta))
    n0, d = kc0.shape
    T = q.shape[0]
    kc = np.zeros((n0 + T, d))
    vc = np.zeros((n0 + T, d))
    kc[:n0] = kc0
    vc[:n0] = vc0
    o = np.empty((T, d))
    lse = np.empty(T)
    fn = _load().path_oracle_decode_vt if value_transport else _load().path_oracle_decode
    fn(_ptr(kc), _ptr(vc), n0, n0 + T, d, _ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), T, float(scale),
       _ptr(o), _ptr(lse))
    return o, lse, kc, vc


def kcache_update(kc, w, beta):
    """Apply (I - beta w w^T) to every row of kc ([n, d]); returns a new array."""
    kc = _f64(kc).copy()
    w = _f64(w)
    n, d = kc.shape
    _load().path_oracle_kcache_update(_ptr(kc), n, d, _ptr(w), float(beta))
    return kc


def path_attn_bwd(q, k, v, w, beta, dO, log_f=None, scale=None):
    """Gradients of causal PaTH(-FoX) attention in fp64, by the chain rule through the walk.

    q, k, v, w, dO: [..., L, d]; beta, log_f: [..., L].  dO is the gradient of the caller's loss
    with respect to o.  Returns dict with dq, dk, dv, dw (shape of q), dbeta (shape of beta) and,
    with log_f, dlog_f.
    """
    q, k, v, w, beta, dO = (_f64(x) for x in (q, k, v, w, beta, dO))
    lf = None if log_f is None else _f64(log_f)
    L, d = q.shape[-2], q.shape[-1]
    BH = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    for x in (k, v, w, dO):
        assert x.shape == q.shape
    assert beta.shape == q.shape[:-1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = {n: np.empty(q.shape) for n in ("dq", "dk", "dv", "dw")}
    out["dbeta"] = np.empty(beta.shape)
    dlf = np.empty(beta.shape) if lf is not None else None
    _load().path_oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(lf), _ptr(dO), BH, L, d,
                            float(scale), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dw"]),
                            _ptr(out["dbeta"]), _ptr(dlf))
    if dlf is not None:
        out["dlog_f"] = dlf
    return out
