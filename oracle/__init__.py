"""CPU fp64 oracle for the KDA backward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
library's product path never touches it and shares no code with it.

``kda_oracle.c`` holds the token-serial recurrence and its hand-derived
reverse mode (see the header of that file for the definition and the
readings of the pages it follows).  ``chunked.py`` holds a second,
independent fp64 restatement in the chunked (WY / UT-transform) form, used
only to pin the chunk algebra against the token-serial definition.

Arrays are numpy float64, token-major ``[Ttot, H, D]`` with sequences packed
back to back (``cu_seqlens``); fixed-length ``[B, T, H, D]`` data is the same
memory with ``cu_seqlens = [0, T, 2T, ...]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int64)),
        ("H", ctypes.c_int),
        ("K", ctypes.c_int),
        ("V", ctypes.c_int),
        ("scale", ctypes.c_double),
        ("eps", ctypes.c_double),
        ("gate_mode", ctypes.c_int),
        ("erase", ctypes.c_int),
        ("normalize", ctypes.c_int),
        ("chunk", ctypes.c_int),
        ("nthreads", ctypes.c_int),
        ("dt_bias", ctypes.POINTER(ctypes.c_double)),
    ]


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``oracle/_build/libkda_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_forward.argtypes = [ctypes.POINTER(_Cfg)] + [dp] * 10
            lib.kda_oracle_forward.restype = ctypes.c_int
            lib.kda_oracle_backward.argtypes = [ctypes.POINTER(_Cfg)] + [dp] * 18
            lib.kda_oracle_backward.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _cfg(cu_seqlens, H, K, V, scale, eps, gate_mode, erase, normalize, chunk,
         nthreads, dt_bias=None):
    """The C config; returns it with the arrays it points at (keep them alive)."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    db = None if dt_bias is None else _f64(np.reshape(dt_bias, (H, K)))
    c = _Cfg(len(cu) - 1, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
             H, K, V, float(scale), float(eps), int(gate_mode), int(erase),
             int(normalize), int(chunk), int(nthreads), _ptr(db))
    return c, (cu, db)


def num_chunks(cu_seqlens, chunk):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = cu[1:] - cu[:-1]
    return int(np.sum((lens + chunk - 1) // chunk))


def forward(q, k, v, g, beta, A_log, h0=None, *, cu_seqlens, scale=None,
            eps=1e-6, gate_mode=0, erase=1, normalize=1, chunk=64,
            want_chunk_states=False, nthreads=0, dt_bias=None):
    """Token-serial fp64 forward.

    Returns ``(o, hT, chunk_states)``; ``chunk_states`` is ``[NTc, H, K, V]``
    (the state at the start of every chunk) or ``None``.
    """
    q, k, v, g, beta, A_log, h0 = map(_f64, (q, k, v, g, beta, A_log, h0))
    Ttot, H, K = q.shape
    V = v.shape[2]
    if scale is None:
        scale = K ** -0.5
    c, keep = _cfg(cu_seqlens, H, K, V, scale, eps, gate_mode, erase, normalize,
                   chunk, nthreads, dt_bias)
    cu = keep[0]
    N = len(cu) - 1
    o = np.zeros((Ttot, H, V))
    hT = np.zeros((N, H, K, V))
    cs = np.zeros((num_chunks(cu, chunk), H, K, V)) if want_chunk_states else None
    rc = _load().kda_oracle_forward(
        ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(A_log), _ptr(h0), _ptr(o), _ptr(hT), _ptr(cs))
    if rc != 0:
        raise ValueError(f"kda_oracle_forward failed ({rc})")
    return o, hT, cs


def backward(q, k, v, g, beta, A_log, h0, dO, dhT, *, cu_seqlens, scale=None,
             eps=1e-6, gate_mode=0, erase=1, normalize=1, chunk=64,
             want_chunk_dstates=False, nthreads=0, dt_bias=None):
    """Token-serial fp64 backward.

    ``dt_bias`` (optional, ``[H, K]``) is the gate's per-channel bias,
    ``gk = -exp(A_log) softplus(g + dt_bias)``.
    Returns a dict with ``dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0`` and, if asked,
    ``chunk_dstates`` ``[NTc, H, K, V]`` (the adjoint of the state at the end
    of every chunk).
    """
    q, k, v, g, beta, A_log, h0, dO, dhT = map(
        _f64, (q, k, v, g, beta, A_log, h0, dO, dhT))
    Ttot, H, K = q.shape
    V = v.shape[2]
    if scale is None:
        scale = K ** -0.5
    c, keep = _cfg(cu_seqlens, H, K, V, scale, eps, gate_mode, erase, normalize,
                   chunk, nthreads, dt_bias)
    cu = keep[0]
    N = len(cu) - 1
    out = dict(
        dq=np.zeros((Ttot, H, K)), dk=np.zeros((Ttot, H, K)),
        dv=np.zeros((Ttot, H, V)), dg=np.zeros((Ttot, H, K)),
        dbeta=np.zeros((Ttot, H)), dA_log=np.zeros((H,)), ddt_bias=np.zeros((H, K)),
        dh0=np.zeros((N, H, K, V)))
    cds = np.zeros((num_chunks(cu, chunk), H, K, V)) if want_chunk_dstates else None
    rc = _load().kda_oracle_backward(
        ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        _ptr(A_log), _ptr(h0), _ptr(dO), _ptr(dhT), _ptr(out["dq"]),
        _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
        _ptr(out["dA_log"]), _ptr(out["ddt_bias"]), _ptr(out["dh0"]), _ptr(cds))
    if rc != 0:
        raise ValueError(f"kda_oracle_backward failed ({rc})")
    if want_chunk_dstates:
        out["chunk_dstates"] = cds
    return out
