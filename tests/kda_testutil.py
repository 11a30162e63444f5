"""Shared helpers of the test-suite: oracle runs on workload inputs, the
per-tensor relative L2 error, and GPU runs through the C ABI."""
import numpy as np
import torch

import oracle
from linear_attention_backward_gb300 import workloads as wl

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "dh0")


def f64_tokens(t):
    """[B, T, H, ...] torch tensor -> fp64 numpy [B*T, H, ...]."""
    return t.double().reshape(-1, *t.shape[2:]).numpy()


def _bias(x):
    b = x.get("dt_bias")
    return None if b is None else b.double().numpy()


def oracle_bwd(x, **kw):
    return oracle.backward(
        f64_tokens(x["q"]), f64_tokens(x["k"]), f64_tokens(x["v"]), f64_tokens(x["g"]),
        f64_tokens(x["beta"]), x["A_log"].double().numpy(), x["h0"].double().numpy(),
        f64_tokens(x["dO"]), x["dhT"].double().numpy(), cu_seqlens=wl.seq_bounds(x),
        dt_bias=_bias(x), **kw)


def oracle_states(x, chunk=64):
    _, hT, cs = oracle.forward(
        f64_tokens(x["q"]), f64_tokens(x["k"]), f64_tokens(x["v"]), f64_tokens(x["g"]),
        f64_tokens(x["beta"]), x["A_log"].double().numpy(), x["h0"].double().numpy(),
        cu_seqlens=wl.seq_bounds(x), chunk=chunk, want_chunk_states=True, dt_bias=_bias(x))
    return cs, hT


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nr = np.linalg.norm(ref)
    d = np.linalg.norm(got - ref)
    return d / nr if nr > 0 else d


def to_dev(x, dev="cuda"):
    return {n: (t.to(dev) if t is not None else None) for n, t in x.items()}


def gpu_bwd(x, states=None, **kw):
    import linear_attention_backward_gb300 as kda
    d = to_dev(x)
    g = kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"], d["dO"],
                d["dhT"], cu_seqlens=d["cu_seqlens"], states=states, dt_bias=d.get("dt_bias"),
                **kw)
    torch.cuda.synchronize()
    return g, d


def slot_index(x, chunk=64):
    """(sequence, chunk) -> slot for the library's slot map, as a list of
    arrays of slots per sequence (dense oracle chunk order = concatenation)."""
    cu = wl.seq_bounds(x)
    out = []
    fixed = x["cu_seqlens"] is None
    T = x["q"].shape[1]
    nps = (T + chunk - 1) // chunk
    for s in range(len(cu) - 1):
        L = cu[s + 1] - cu[s]
        n = (L + chunk - 1) // chunk
        base = s * nps if fixed else cu[s] // chunk + s
        out.append(np.arange(base, base + n))
    return out


def unpack_core_tiles(t):
    """[..., 128, 128] tiles in packed core-matrix order (8 x 8 cores, cores
    along the second axis first) -> row-major, as a new tensor."""
    lead = t.shape[:-2]
    R, C = t.shape[-2], t.shape[-1]
    x = t.reshape(*lead, R // 8, C // 8, 8, 8)
    return x.transpose(-3, -2).reshape(*lead, R, C).contiguous()


def check_dalog(g, ref, x, tol):
    """dA_log[h] sums dgk * gk over every token and channel of head h, terms
    of both signs: its error is that of the terms (per-tensor tol, as dg)
    times the cancellation ||terms||_2 / |sum|.  Bounded here against the
    L2 norm of the oracle's terms, per head (dgk * gk = dg softplus / sigmoid
    of the biased gate)."""
    z = f64_tokens(x["g"]) + (0.0 if x.get("dt_bias") is None
                              else x["dt_bias"].double().numpy()[None])
    terms = ref["dg"] * np.logaddexp(0.0, z) * (1.0 + np.exp(-z))
    got = g["dA_log"].double().cpu().numpy()
    for h in range(got.shape[0]):
        l2 = np.linalg.norm(terms[:, h])
        assert abs(got[h] - ref["dA_log"][h]) <= tol * l2, (h, got[h], ref["dA_log"][h], l2)
