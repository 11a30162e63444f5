"""Python binding of the GB300 KDA backward library (``libkda.so``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI of ``include/kda.h``.  PyTorch provides device
memory (outputs and the workspace are ``torch.empty`` buffers) and the stream
(``torch.cuda.current_stream()``).  There is no CPU fallback: if the compiled
library is missing, importing the binding's functions raises.

Layouts (all contiguous, token-major): q, k, g ``[B, T, H, K]``; v, dO
``[B, T, H, V]``; beta ``[B, T, H]``; A_log ``[H]`` fp32; h0 / dh_T / dh0
``[N, H, K, V]`` fp32.  Varlen batches pass ``cu_seqlens`` (int32 CUDA tensor
``[N + 1]``) with B = 1.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libkda.so")

KDA_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace",
                4: "cuda error", 5: "timeout", 6: "bad cu_seqlens on device",
                7: "too large for the no-allocation scratch", 8: "gate beyond the block range"}
KDA_FP32, KDA_BF16 = 0, 1


class KdaError(RuntimeError):
    def __init__(self, status, where):
        super().__init__(f"{where}: kda status {status} ({STATUS_NAMES.get(status, '?')})")
        self.status = status


class KdaShape(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
        ("K", ctypes.c_int), ("V", ctypes.c_int), ("chunk", ctypes.c_int),
        ("num_seqs", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p),
        ("scale", ctypes.c_float), ("l2_eps", ctypes.c_float), ("dtype", ctypes.c_int),
    ]


_lib = None
_VP = ctypes.c_void_p


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded ``libkda.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"libkda.so not built ({_LIB_PATH}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(_LIB_PATH)
        S = ctypes.POINTER(KdaShape)
        L.kda_num_chunk_slots.argtypes = [S]
        L.kda_num_chunk_slots.restype = ctypes.c_int64
        L.kda_workspace_bytes.argtypes = [S]
        L.kda_workspace_bytes.restype = ctypes.c_size_t
        L.kda_workspace_dstates_offset.argtypes = [S]
        L.kda_workspace_dstates_offset.restype = ctypes.c_size_t
        L.kda_scan_segments.argtypes = [S]
        L.kda_scan_segments.restype = ctypes.c_int
        L.kda_fwd_states.argtypes = [S] + [_VP] * 11 + [ctypes.c_size_t, _VP]
        L.kda_fwd_states.restype = ctypes.c_int
        L.kda_fwd.argtypes = [S] + [_VP] * 11 + [ctypes.c_size_t, _VP]
        L.kda_fwd.restype = ctypes.c_int
        L.kda_bwd.argtypes = [S] + [_VP] * 20 + [ctypes.c_size_t, _VP]
        L.kda_bwd.restype = ctypes.c_int
        L.kda_bwd_timed.argtypes = [S] + [_VP] * 20 + [ctypes.c_size_t, _VP, _VP]
        L.kda_bwd_timed.restype = ctypes.c_int
        L.kda_bwd_noalloc.argtypes = [S] + [_VP] * 18 + [_VP]
        L.kda_bwd_noalloc.restype = ctypes.c_int
        L.kda_noalloc_scratch_bytes.argtypes = []
        L.kda_noalloc_scratch_bytes.restype = ctypes.c_size_t
        L.kda_get_device_status.argtypes = [_VP]
        L.kda_get_device_status.restype = ctypes.c_int
        L.kda_check_cu_seqlens_host.argtypes = [_VP, ctypes.c_int, ctypes.c_int]
        L.kda_check_cu_seqlens_host.restype = ctypes.c_int
        L.kda_status_str.argtypes = [ctypes.c_int]
        L.kda_status_str.restype = ctypes.c_char_p
        L.kda_abi_version.argtypes = []
        L.kda_abi_version.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def make_shape(q_or_k, v, *, cu_seqlens=None, scale=None, l2_eps=None, chunk=64) -> KdaShape:
    B, T, H, K = q_or_k.shape
    V = v.shape[-1]
    dt = {torch.float32: KDA_FP32, torch.bfloat16: KDA_BF16}.get(q_or_k.dtype)
    if dt is None:
        raise TypeError(f"unsupported dtype {q_or_k.dtype}")
    ns = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    return KdaShape(B, T, H, K, V, chunk, ns,
                    None if cu_seqlens is None else cu_seqlens.data_ptr(),
                    float(scale) if scale is not None else 0.0,
                    float(l2_eps) if l2_eps is not None else -1.0, dt)


def num_chunk_slots(shape: KdaShape) -> int:
    return int(lib().kda_num_chunk_slots(ctypes.byref(shape)))


def workspace_bytes(shape: KdaShape) -> int:
    return int(lib().kda_workspace_bytes(ctypes.byref(shape)))


def workspace_dstates_offset(shape: KdaShape) -> int:
    return int(lib().kda_workspace_dstates_offset(ctypes.byref(shape)))


def scan_segments(shape: KdaShape) -> int:
    """Segments of the context-parallel state scans for this shape (0: none)."""
    return int(lib().kda_scan_segments(ctypes.byref(shape)))


def check_cu_seqlens_host(cu_seqlens_cpu: torch.Tensor, total_T: int) -> int:
    cu = cu_seqlens_cpu.to(torch.int32).contiguous()
    return int(lib().kda_check_cu_seqlens_host(ctypes.c_void_p(cu.data_ptr()),
                                               cu.numel() - 1, int(total_T)))


def get_device_status() -> int:
    return int(lib().kda_get_device_status(_stream()))


def _check(st, where):
    if st != KDA_OK:
        raise KdaError(st, where)


def _nseq(B, cu_seqlens):
    return B if cu_seqlens is None else cu_seqlens.numel() - 1


def fwd_states(q, k, v, g, beta, A_log, h0=None, *, cu_seqlens=None, scale=None, l2_eps=None,
               states=None, hT=None, want_hT=False, dt_bias=None, workspace=None):
    """Chunk-start states ``[slots, H, K, V]`` (dtype of k) and optionally hT.

    For bf16 with K = V = 128 every K x V tile is in packed core-matrix order
    (see ``kda_fwd_states`` in include/kda.h; ``unpack_core_tiles`` in the
    tests turns it row-major), the layout :func:`bwd` takes back as
    ``states``.  For bf16 (K = V = 128 or 64) ``workspace`` (uint8 CUDA
    tensor of at least ``workspace_bytes``) is allocated when not given.
    Other shapes return row-major tiles and use no workspace."""
    shape = make_shape(k, v, cu_seqlens=cu_seqlens, scale=scale, l2_eps=l2_eps)
    B, T, H, K = k.shape
    V = v.shape[-1]
    if states is None:
        states = torch.empty((num_chunk_slots(shape), H, K, V), dtype=k.dtype, device=k.device)
    if want_hT and hT is None:
        hT = torch.empty((_nseq(B, cu_seqlens), H, K, V), dtype=torch.float32, device=k.device)
    tc = k.dtype == torch.bfloat16 and K == V and K in (64, 128)
    if workspace is None and tc:
        workspace = torch.empty((workspace_bytes(shape),), dtype=torch.uint8, device=k.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().kda_fwd_states(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                              _ptr(beta), _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(states),
                              _ptr(hT), _ptr(workspace), ctypes.c_size_t(nbytes), _stream())
    _check(st, "kda_fwd_states")
    return (states, hT) if want_hT else states


def fwd(q, k, v, g, beta, A_log, h0=None, *, cu_seqlens=None, scale=None, l2_eps=None,
        o=None, hT=None, want_hT=False, workspace=None, dt_bias=None):
    """Forward read-out ``o`` [B, T, H, V] (bf16, K = V = 128 or 64) and, if asked,
    the final states ``hT`` [N, H, K, V] fp32: ``(o, hT)`` or ``o``.
    ``dt_bias`` (optional fp32 [H, K]) is the gate's per-channel bias."""
    shape = make_shape(q, v, cu_seqlens=cu_seqlens, scale=scale, l2_eps=l2_eps)
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    if o is None:
        o = torch.empty((B, T, H, V), dtype=v.dtype, device=dev)
    if want_hT and hT is None:
        hT = torch.empty((_nseq(B, cu_seqlens), H, K, V), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty((workspace_bytes(shape),), dtype=torch.uint8, device=dev)
    st = lib().kda_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                       _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(o), _ptr(hT),
                       _ptr(workspace),
                       ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream())
    _check(st, "kda_fwd")
    return (o, hT) if want_hT else o


def bwd(q, k, v, g, beta, A_log, h0, dO, dh_T=None, *, cu_seqlens=None, scale=None,
        l2_eps=None, states=None, out=None, workspace=None, events=None, dt_bias=None):
    """Gradients ``dict(dq, dk, dv, dg, dbeta, dA_log, dh0)``, plus ``ddt_bias``
    [H, K] fp32 when ``dt_bias`` (the gate's per-channel bias) is given.

    ``out`` may hold preallocated output tensors under the same keys and
    ``workspace`` a uint8 CUDA tensor of at least ``workspace_bytes`` bytes.
    ``states`` (optional) are :func:`fwd_states`' output for the same inputs,
    in its layout.
    ``events``: optional 5 ``torch.cuda.Event(enable_timing=True)`` recorded at
    the phase boundaries (see ``kda_bwd_timed`` in include/kda.h).
    """
    shape = make_shape(q, v, cu_seqlens=cu_seqlens, scale=scale, l2_eps=l2_eps)
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    if out is None:
        out = {}
    o = dict(out)
    o.setdefault("dq", torch.empty_like(q))
    o.setdefault("dk", torch.empty_like(k))
    o.setdefault("dv", torch.empty_like(v))
    o.setdefault("dg", torch.empty_like(g))
    o.setdefault("dbeta", torch.empty_like(beta))
    o.setdefault("dA_log", torch.empty((H,), dtype=torch.float32, device=dev))
    if dt_bias is not None:
        o.setdefault("ddt_bias", torch.empty((H, K), dtype=torch.float32, device=dev))
    o.setdefault("dh0", torch.empty((_nseq(B, cu_seqlens), H, K, V), dtype=torch.float32,
                                    device=dev))
    need = workspace_bytes(shape)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=dev)
    ev = None
    if events is not None:
        if len(events) != 5:
            raise ValueError("events: 5 timing events expected")
        ev = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    st = lib().kda_bwd_timed(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                             _ptr(beta), _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(dO),
                             _ptr(dh_T), _ptr(o["dq"]), _ptr(o["dk"]), _ptr(o["dv"]),
                             _ptr(o["dg"]), _ptr(o["dbeta"]), _ptr(o["dA_log"]),
                             _ptr(o.get("ddt_bias")), _ptr(o["dh0"]),
                             _ptr(states), _ptr(workspace),
                             ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                             _stream(), ev)
    _check(st, "kda_bwd")
    o["_workspace"] = workspace
    return o


def noalloc_scratch_bytes() -> int:
    """Capacity of the fixed scratch array used by :func:`bwd_noalloc`."""
    return int(lib().kda_noalloc_scratch_bytes())


def bwd_noalloc(q, k, v, g, beta, A_log, h0, dO, dh_T=None, *, out, cu_seqlens=None,
                scale=None, l2_eps=None, dt_bias=None):
    """Backward pass through ``kda_bwd_noalloc``: for callers that cannot
    allocate device memory, the library uses its own fixed scratch array
    instead of a caller workspace.  ``out`` must hold preallocated dq, dk,
    dv, dg, dbeta, dA_log and dh0 (and ddt_bias for a ``dt_bias``); nothing is
    allocated here.  Raises
    KdaError(7) when the problem does not fit the scratch array."""
    shape = make_shape(q, v, cu_seqlens=cu_seqlens, scale=scale, l2_eps=l2_eps)
    st = lib().kda_bwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                               _ptr(beta), _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(dO),
                               _ptr(dh_T), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                               _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["dA_log"]),
                               _ptr(out.get("ddt_bias")), _ptr(out.get("dh0")), _stream())
    _check(st, "kda_bwd_noalloc")
    return out


class KDAFunction(torch.autograd.Function):
    """Differentiable KDA layer core: ``(o, hT) = KDAFunction.apply(q, k, v, g,
    beta, A_log, h0, dt_bias, cu_seqlens, scale, l2_eps)``.  The forward is
    :func:`fwd` (bf16, K = V = 128) and the backward :func:`bwd`, which
    recomputes the chunk states from the saved inputs.  Gradients flow to q,
    k, v, g, beta, A_log and, where given, h0 and dt_bias."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, A_log, h0, dt_bias, cu_seqlens, scale, l2_eps):
        o, hT = fwd(q, k, v, g, beta, A_log, h0, cu_seqlens=cu_seqlens, scale=scale,
                    l2_eps=l2_eps, want_hT=True, dt_bias=dt_bias)
        ctx.save_for_backward(q, k, v, g, beta, A_log, h0, dt_bias, cu_seqlens)
        ctx.scale, ctx.l2_eps = scale, l2_eps
        return o, hT

    @staticmethod
    def backward(ctx, dO, dhT):
        q, k, v, g, beta, A_log, h0, dt_bias, cu_seqlens = ctx.saved_tensors
        if dO is None:
            dO = torch.zeros_like(v)
        gr = bwd(q, k, v, g, beta, A_log, h0, dO.contiguous(),
                 None if dhT is None else dhT.contiguous(), cu_seqlens=cu_seqlens,
                 scale=ctx.scale, l2_eps=ctx.l2_eps, dt_bias=dt_bias)
        return (gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], gr["dA_log"],
                gr["dh0"] if h0 is not None else None,
                gr.get("ddt_bias") if dt_bias is not None else None, None, None, None)


def kda(q, k, v, g, beta, A_log, h0=None, *, dt_bias=None, cu_seqlens=None, scale=None,
        l2_eps=None):
    """The differentiable forward ``(o, hT)`` through :class:`KDAFunction`."""
    return KDAFunction.apply(q, k, v, g, beta, A_log, h0, dt_bias, cu_seqlens, scale, l2_eps)
