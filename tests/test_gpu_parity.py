"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle,
element by element, per-tensor relative L2.  Tolerances: 1e-4 for fp32
inputs, 2e-2 for bf16 inputs (bf16 operands, fp32 accumulation)."""
import numpy as np
import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda
from linear_attention_backward_gb300 import workloads as wl
from kda_testutil import (GRADS, check_dalog as _check_dalog, f64_tokens, gpu_bwd, oracle_bwd,
                          oracle_states, rel_l2,
                          unpack_core_tiles,
                          slot_index)

pytestmark = pytest.mark.gpu

TOL = {"fp32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _compare(g, ref, x, tol, keys=GRADS):
    errs = {}
    for key in keys:
        got = g[key].double().cpu().numpy().reshape(ref[key].shape)
        errs[key] = rel_l2(got, ref[key])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"rel-L2 above {tol}: {bad} (all: {errs})"
    return errs


def _check_status():
    assert kda.get_device_status() == 0


def test_tiny_fp32_workload():
    w = wl.WORKLOADS["tiny_fp32"]
    x = wl.make_inputs(w)
    g, _ = gpu_bwd(x)
    _check_status()
    _compare(g, oracle_bwd(x), x, TOL["fp32"])


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("T", [1, 63, 65, 200])
def test_bf16_fixed_ragged(K, T):
    w = wl.custom("t", B=2, T=T, H=2, K=K, V=K, dtype="bf16", with_h0=True, with_dhT=True)
    x = wl.make_inputs(w, seed=T + K)
    g, _ = gpu_bwd(x)
    _check_status()
    _compare(g, oracle_bwd(x), x, TOL["bf16"])


@pytest.mark.parametrize("T", [1, 77, 256])
def test_fp32_ragged_with_states(T):
    w = wl.custom("t", B=2, T=T, H=2, K=64, V=64, dtype="fp32", with_h0=True, with_dhT=True)
    x = wl.make_inputs(w, seed=3 + T)
    g, _ = gpu_bwd(x)
    _check_status()
    _compare(g, oracle_bwd(x), x, TOL["fp32"])


def test_varlen_bf16_with_empty_sequence():
    w = wl.custom("v", H=2, K=128, V=128, dtype="bf16", with_h0=True, with_dhT=True,
                  varlen=(5, 1, 200))
    lengths = [1, 63, 0, 130, 65]
    x = wl.make_inputs(w, seed=5, lengths=lengths)
    assert kda.check_cu_seqlens_host(x["cu_seqlens"], int(x["cu_seqlens"][-1])) == 0
    g, _ = gpu_bwd(x)
    _check_status()
    ref = oracle_bwd(x)
    _compare(g, ref, x, TOL["bf16"])
    # the empty sequence passes its state gradient straight through
    np.testing.assert_allclose(g["dh0"][2].cpu().numpy(), x["dhT"][2].numpy(), rtol=0, atol=0)


def _with_bias(x, seed):
    H, K = x["q"].shape[2], x["q"].shape[3]
    gen = torch.Generator().manual_seed(seed)
    return dict(x, dt_bias=torch.randn(H, K, generator=gen) * 0.5)


@pytest.mark.parametrize("dtype,K,T", [("bf16", 128, 200), ("bf16", 64, 130), ("fp32", 64, 97)])
def test_gate_bias(dtype, K, T):
    # gk = -exp(A_log) softplus(g + dt_bias) and its gradient ddt_bias, on the
    # tcgen05 path (bf16, K = 128) and the mma.sync paths
    w = wl.custom("gb", B=2, T=T, H=2, K=K, V=K, dtype=dtype, with_h0=True, with_dhT=True)
    x = _with_bias(wl.make_inputs(w, seed=31 + T), 5)
    g, _ = gpu_bwd(x)
    _check_status()
    ref = oracle_bwd(x)
    keys = tuple(k for k in GRADS if k != "dA_log") + ("ddt_bias",)
    _compare(g, ref, x, TOL[dtype], keys=keys)
    _check_dalog(g, ref, x, TOL[dtype])


def test_gate_bias_varlen():
    lengths = [64, 0, 130, 1, 70]
    w = wl.custom("gbv", H=2, K=128, V=128, dtype="bf16", with_h0=True, with_dhT=True,
                  varlen=(5, 0, 256))
    x = _with_bias(wl.make_inputs(w, seed=12, lengths=lengths), 6)
    g, _ = gpu_bwd(x)
    _check_status()
    ref = oracle_bwd(x)
    keys = tuple(k for k in GRADS if k != "dA_log") + ("ddt_bias",)
    _compare(g, ref, x, TOL["bf16"], keys=keys)
    _check_dalog(g, ref, x, TOL["bf16"])


def test_varlen_many_sequences_with_ties():
    # the scans take the sequences longest first: equal lengths (ties broken by
    # index), empty sequences and more sequences than one wave of scan CTAs
    lengths = [64, 0, 130, 64, 1, 200, 130, 0, 63, 64, 129, 5] * 4
    w = wl.custom("vt", H=2, K=128, V=128, dtype="bf16", with_h0=True, with_dhT=True,
                  varlen=(len(lengths), 0, 256))
    x = wl.make_inputs(w, seed=11, lengths=lengths)
    g, _ = gpu_bwd(x)
    _check_status()
    _compare(g, oracle_bwd(x), x, TOL["bf16"])


def test_fwd_states_and_reverse_scan_intermediates():
    w = wl.custom("s", B=2, T=190, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=9)
    d = {n: (t.cuda() if t is not None else None) for n, t in x.items()}
    states, hT = kda.fwd_states(d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                                want_hT=True)
    torch.cuda.synchronize()
    cs, hT_ref = oracle_states(x)
    slots = np.concatenate(slot_index(x))
    got = states.double().cpu().numpy()[slots]
    assert rel_l2(got, cs) < 1e-2
    assert rel_l2(hT.double().cpu().numpy(), hT_ref) < 1e-2
    # reverse scan: dS at every chunk end, read from the documented workspace offset
    g = kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"], d["dO"],
                d["dhT"])
    torch.cuda.synchronize()
    shape = kda.make_shape(d["q"], d["v"])
    off = kda.workspace_dstates_offset(shape)
    n = kda.num_chunk_slots(shape) * 2 * 128 * 128
    ws = g["_workspace"]
    # bf16 K = V = 128: tiles in packed core-matrix order (include/kda.h)
    dst = unpack_core_tiles(ws[off:off + 2 * n].view(torch.bfloat16).reshape(-1, 2, 128, 128))
    ref = oracle_bwd(x, want_chunk_dstates=True)
    assert rel_l2(dst.double().cpu().numpy()[slots], ref["chunk_dstates"]) < 1e-2
    # forward states recomputed inside kda_bwd (start of the workspace)
    ins = unpack_core_tiles(ws[:2 * n].view(torch.bfloat16).reshape(-1, 2, 128, 128))
    assert rel_l2(ins.double().cpu().numpy()[slots], cs) < 1e-2


def test_states_given_matches_internal_recompute():
    w = wl.custom("s", B=1, T=300, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=4)
    g1, d = gpu_bwd(x)
    torch.cuda.synchronize()
    shape = kda.make_shape(d["q"], d["v"])
    n = kda.num_chunk_slots(shape) * 2 * 128 * 128
    # the recomputed states sit at the start of the workspace; handing the same
    # bf16 states back must reproduce every gradient bit for bit
    internal = unpack_core_tiles(
        g1["_workspace"][:2 * n].view(torch.bfloat16).reshape(-1, 2, 128, 128))
    g2, _ = gpu_bwd(x, states=internal)
    for key in GRADS:
        assert torch.equal(g1[key], g2[key]), key
    # kda_fwd_states computes the same states by its own scan (rounding-level
    # differences only), and gradients from them stay within the tolerance
    states = kda.fwd_states(d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"])
    slots = np.concatenate(slot_index(x))
    a = states.double().cpu().numpy()[slots]
    b = internal.double().cpu().numpy()[slots]
    assert rel_l2(a, b) < 5e-3
    g3, _ = gpu_bwd(x, states=states)
    ref = oracle_bwd(x)
    _compare(g3, ref, x, TOL["bf16"])


def test_states_given_with_gate_bias():
    # kda_fwd_states with the gate bias feeds kda_bwd with the same bias
    w = wl.custom("sb", B=2, T=170, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = _with_bias(wl.make_inputs(w, seed=14), 9)
    d = {n: (t.cuda() if t is not None else None) for n, t in x.items()}
    states = kda.fwd_states(d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                            dt_bias=d["dt_bias"])
    g, _ = gpu_bwd(x, states=states)
    _check_status()
    ref = oracle_bwd(x)
    keys = tuple(k for k in GRADS if k != "dA_log") + ("ddt_bias",)
    _compare(g, ref, x, TOL["bf16"], keys=keys)
    _check_dalog(g, ref, x, TOL["bf16"])


def test_repeatable_bitwise():
    w = wl.custom("r", B=2, T=256, H=4, K=128, V=128, dtype="bf16")
    x = wl.make_inputs(w, seed=2)
    g1, _ = gpu_bwd(x)
    g2, _ = gpu_bwd(x)
    for key in GRADS:
        assert torch.equal(g1[key], g2[key]), key


def test_outputs_do_not_spill_past_their_rows():
    """Outputs live in the front of larger canary-filled buffers; nothing past
    the valid tokens (ragged last chunk, varlen tail) may be written."""
    w = wl.custom("c", H=2, K=128, V=128, dtype="bf16", varlen=(3, 1, 100))
    x = wl.make_inputs(w, seed=8, lengths=[70, 5, 58])
    d = {n: (t.cuda() if t is not None else None) for n, t in x.items()}
    T = x["q"].shape[1]
    out, bigs = {}, {}
    for key, like in (("dq", d["q"]), ("dk", d["k"]), ("dv", d["v"]), ("dg", d["g"]),
                      ("dbeta", d["beta"])):
        n = like.numel()
        big = torch.full((n + 4096,), 7.0, dtype=like.dtype, device="cuda")
        bigs[key] = (big, n)
        out[key] = big[:n].view(like.shape)
    kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"], d["dO"], d["dhT"],
            cu_seqlens=d["cu_seqlens"], out=out)
    torch.cuda.synchronize()
    for key, (big, n) in bigs.items():
        assert torch.all(big[n:] == 7.0), key
    assert T == 133


# ---------------------------------------------------------------------------
# Full-size workloads in the benchmark's launch configuration: the whole
# backward runs on the GPU; the oracle checks sampled (sequence, head) units.
# ---------------------------------------------------------------------------
def _sample_units(x, units, dalog_head=None):
    """Run the oracle on (sequence, head) units only.  Returns, per unit, the
    oracle's grads; and dA_log for `dalog_head` summed over all sequences."""
    cu = wl.seq_bounds(x)
    out = {}
    for (s, h) in units:
        a, b = cu[s], cu[s + 1]
        sub = {}
        for n in ("q", "k", "v", "g", "dO"):
            sub[n] = x[n].reshape(-1, *x[n].shape[2:])[a:b, h:h + 1].unsqueeze(0)
        sub["beta"] = x["beta"].reshape(-1, x["beta"].shape[-1])[a:b, h:h + 1].unsqueeze(0)
        sub["A_log"] = x["A_log"][h:h + 1]
        sub["h0"] = x["h0"][s:s + 1, h:h + 1]
        sub["dhT"] = x["dhT"][s:s + 1, h:h + 1]
        sub["cu_seqlens"] = None
        out[(s, h)] = oracle_bwd(sub, nthreads=0)
    dA = None
    if dalog_head is not None:
        h = dalog_head
        total = 0.0
        seqs = list(range(len(cu) - 1))
        for s in seqs:
            if (s, h) in out:
                total += out[(s, h)]["dA_log"][0]
        missing = [s for s in seqs if (s, h) not in out]
        if missing:
            # all remaining sequences of that head in one oracle call (threads over sequences)
            import oracle as orc
            flat = lambda t: t.reshape(-1, *t.shape[2:])
            sel = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in missing])
            cu2 = np.concatenate([[0], np.cumsum([cu[s + 1] - cu[s] for s in missing])])
            pick = lambda t: flat(t)[sel][:, h:h + 1].double().numpy()
            r = orc.backward(pick(x["q"]), pick(x["k"]), pick(x["v"]), pick(x["g"]),
                             flat(x["beta"])[sel][:, h:h + 1].double().numpy(),
                             x["A_log"][h:h + 1].double().numpy(),
                             x["h0"][missing][:, h:h + 1].double().numpy(), pick(x["dO"]),
                             x["dhT"][missing][:, h:h + 1].double().numpy(), cu_seqlens=cu2)
            total += r["dA_log"][0]
        dA = total
    return out, dA


@pytest.mark.parametrize("name,units,dalog_head", [
    ("lowpar_bf16", [(0, 0), (0, 15)], 3),
    ("main_bf16", [(0, 0), (3, 31), (2, 17)], 5),
    ("large_bf16", [(7, 31), (0, 1)], None),
    ("varlen_bf16", [(0, 0), (6, 12), (15, 31)], 7),
])
def test_full_size_sampled(name, units, dalog_head):
    w = wl.WORKLOADS[name]
    x = wl.make_inputs(w)
    g, _ = gpu_bwd(x)
    _check_status()
    ref, dA = _sample_units(x, units, dalog_head)
    cu = wl.seq_bounds(x)
    errs = {}
    for (s, h), r in ref.items():
        a, b = cu[s], cu[s + 1]
        for key in ("dq", "dk", "dv", "dg"):
            got = g[key].reshape(-1, *g[key].shape[2:])[a:b, h].double().cpu().numpy()
            errs[(s, h, key)] = rel_l2(got, r[key][:, 0])
        got = g["dbeta"].reshape(-1, g["dbeta"].shape[-1])[a:b, h].double().cpu().numpy()
        errs[(s, h, "dbeta")] = rel_l2(got, r["dbeta"][:, 0])
        errs[(s, h, "dh0")] = rel_l2(g["dh0"][s, h].double().cpu().numpy(), r["dh0"][0, 0])
    if dA is not None:
        errs[("dA_log", dalog_head)] = abs(g["dA_log"][dalog_head].item() - dA) / abs(dA)
    bad = {k: v for k, v in errs.items() if not v <= TOL["bf16"]}
    assert not bad, f"{name}: {bad}"
    # properties at full size: every gradient finite
    for key in GRADS:
        assert torch.isfinite(g[key].float()).all(), key


def test_per_band_scans_feed_the_tensor_core_gradients(monkeypatch):
    """KDA_SCAN_LEGACY=1: the per-band scans (row-major states and state
    gradients) in front of the tensor-core gradient kernel."""
    monkeypatch.setenv("KDA_SCAN_LEGACY", "1")
    w = wl.custom("lg", B=2, T=200, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=17)
    g, _ = gpu_bwd(x)
    _compare(g, oracle_bwd(x), x, TOL["bf16"])
