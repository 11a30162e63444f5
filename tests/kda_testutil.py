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


def check_dalog_biased(g, ref, x, tol):
    """WEAKER dA_log check, used only by the gate-bias (dt_bias) tests.

    Every other test compares dA_log by the plain per-tensor relative L2
    bound over the [H] vector, like the other gradients.  With a gate bias
    the sum dA_log[h] = sum dgk * gk cancels by ~20x (terms of both signs),
    so its relative error is that of the terms (the dg error) times the
    cancellation.  Here the per-head error is bounded by tol times the L2
    norm of the oracle's terms (dgk * gk = dg softplus / sigmoid of the
    biased gate) instead of tol times |dA_log[h]|."""
    z = f64_tokens(x["g"]) + (0.0 if x.get("dt_bias") is None
                              else x["dt_bias"].double().numpy()[None])
    terms = ref["dg"] * np.logaddexp(0.0, z) * (1.0 + np.exp(-z))
    got = g["dA_log"].double().cpu().numpy()
    for h in range(got.shape[0]):
        l2 = np.linalg.norm(terms[:, h])
        assert abs(got[h] - ref["dA_log"][h]) <= tol * l2, (h, got[h], ref["dA_log"][h], l2)


def full_parity(x, g, keys=GRADS, nthreads=0):
    """Per-tensor relative L2 error of every gradient over a whole workload.

    The oracle runs one sequence at a time (all heads, OpenMP over heads) so
    that its fp64 arrays stay a fraction of the workload's; the squared norms
    of the error and of the oracle's tensor are summed over sequences, and
    dA_log (a sum over sequences) is summed before it is compared.  ``g``
    holds the GPU gradients (device tensors).  Returns {key: rel-L2}."""
    cu = wl.seq_bounds(x)
    flat = lambda t: t.reshape(-1, *t.shape[2:])
    H = x["q"].shape[2]
    num = {k: 0.0 for k in keys}
    den = {k: 0.0 for k in keys}
    dA = np.zeros(H)
    ddt = None if x.get("dt_bias") is None else np.zeros(tuple(x["dt_bias"].shape))
    tok_keys = [k for k in ("dq", "dk", "dv", "dg", "dbeta") if k in keys]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if b == a:
            ref = {"dh0": x["dhT"][s].double().numpy()}
        else:
            pick = lambda n: flat(x[n])[a:b].double().numpy()
            ref = oracle.backward(
                pick("q"), pick("k"), pick("v"), pick("g"), pick("beta"),
                x["A_log"].double().numpy(), x["h0"][s:s + 1].double().numpy(), pick("dO"),
                x["dhT"][s:s + 1].double().numpy(), cu_seqlens=[0, b - a],
                dt_bias=_bias(x), nthreads=nthreads)
            dA += ref["dA_log"]
            if ddt is not None:
                ddt += ref["ddt_bias"]
            for key in tok_keys:
                got = flat(g[key])[a:b].double().cpu().numpy()
                num[key] += float(np.sum((got - ref[key]) ** 2))
                den[key] += float(np.sum(ref[key] ** 2))
            ref["dh0"] = ref["dh0"][0]
        if "dh0" in keys:
            got = g["dh0"][s].double().cpu().numpy()
            num["dh0"] += float(np.sum((got - ref["dh0"]) ** 2))
            den["dh0"] += float(np.sum(ref["dh0"] ** 2))
    errs = {k: (np.sqrt(num[k] / den[k]) if den[k] > 0 else np.sqrt(num[k]))
            for k in keys if k != "dA_log"}
    if "dA_log" in keys:
        errs["dA_log"] = rel_l2(g["dA_log"].double().cpu().numpy(), dA)
    if ddt is not None and "ddt_bias" in g:
        errs["ddt_bias"] = rel_l2(g["ddt_bias"].double().cpu().numpy(), ddt)
    return errs
