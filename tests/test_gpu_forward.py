"""GPU parity of the forward pass (kda_fwd: the read-out o and the final
states hT) against the fp64 token-serial oracle forward, per-tensor relative
L2 (bf16 inputs: 2e-2), through the C ABI."""
import numpy as np
import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda
import oracle
from linear_attention_backward_gb300 import workloads as wl
from kda_testutil import f64_tokens, rel_l2, to_dev

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()
    assert torch.cuda.is_available()


def oracle_fwd(x):
    b = x.get("dt_bias")
    o, hT, _ = oracle.forward(
        f64_tokens(x["q"]), f64_tokens(x["k"]), f64_tokens(x["v"]), f64_tokens(x["g"]),
        f64_tokens(x["beta"]), x["A_log"].double().numpy(), x["h0"].double().numpy(),
        cu_seqlens=wl.seq_bounds(x), dt_bias=None if b is None else b.double().numpy())
    return o, hT


def gpu_fwd(x):
    d = to_dev(x)
    o, hT = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                    cu_seqlens=d["cu_seqlens"], want_hT=True, dt_bias=d.get("dt_bias"))
    torch.cuda.synchronize()
    assert kda.get_device_status() == 0
    return o, hT


def _check(x, o, hT):
    ro, rhT = oracle_fwd(x)
    got = o.double().cpu().numpy().reshape(ro.shape)
    assert np.isfinite(got).all()
    e_o = rel_l2(got, ro)
    e_h = rel_l2(hT.double().cpu().numpy(), rhT)
    assert e_o <= TOL and e_h <= TOL, (e_o, e_h)
    return e_o, e_h


@pytest.mark.parametrize("T", [64, 200, 321])
def test_fixed_ragged(T):
    # several chunks and a ragged last chunk; nonzero initial state
    w = wl.custom("f", B=2, T=T, H=3, K=128, V=128, dtype="bf16", with_h0=True)
    x = wl.make_inputs(w, seed=21 + T)
    _check(x, *gpu_fwd(x))


def test_gate_bias():
    w = wl.custom("fgb", B=2, T=150, H=2, K=128, V=128, dtype="bf16", with_h0=True)
    x = wl.make_inputs(w, seed=8)
    gen = torch.Generator().manual_seed(3)
    x["dt_bias"] = torch.randn(2, 128, generator=gen) * 0.5
    _check(x, *gpu_fwd(x))


def test_zero_initial_state():
    w = wl.custom("f0", B=1, T=130, H=2, K=128, V=128, dtype="bf16")
    x = wl.make_inputs(w, seed=4)
    _check(x, *gpu_fwd(x))


def test_varlen_with_empty_and_tied_sequences():
    lengths = [64, 0, 130, 64, 1, 200, 0, 63]
    w = wl.custom("fv", H=2, K=128, V=128, dtype="bf16", with_h0=True, varlen=(8, 0, 256))
    x = wl.make_inputs(w, seed=9, lengths=lengths)
    o, hT = gpu_fwd(x)
    _check(x, o, hT)
    # an empty sequence hands its initial state through unchanged
    np.testing.assert_allclose(hT[1].cpu().numpy(), x["h0"][1].numpy(), rtol=0, atol=0)


def test_rows_outside_the_sequences_untouched():
    # o is written on the sequences' rows only: a sentinel in a larger buffer
    w = wl.custom("fs", B=1, T=100, H=2, K=128, V=128, dtype="bf16")
    x = wl.make_inputs(w, seed=2)
    d = to_dev(x)
    big = torch.full((1, 101, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    o = big[:, :100]
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], None, o=o)
    torch.cuda.synchronize()
    assert (big[:, 100] == 7.0).all()
    ro, _ = oracle_fwd(x)
    assert rel_l2(o.double().cpu().numpy().reshape(ro.shape), ro) <= TOL


def test_repeatable_bitwise():
    w = wl.custom("fb", B=1, T=256, H=2, K=128, V=128, dtype="bf16", with_h0=True)
    x = wl.make_inputs(w, seed=13)
    o1, h1 = gpu_fwd(x)
    o2, h2 = gpu_fwd(x)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


@pytest.mark.parametrize("name,units", [("main_bf16", [(0, 0), (3, 31)]),
                                        ("varlen_bf16", [(6, 12), (15, 31)])])
def test_full_size_sampled(name, units):
    w = wl.WORKLOADS[name]
    x = wl.make_inputs(w)
    o, hT = gpu_fwd(x)
    cu = wl.seq_bounds(x)
    flat = lambda t: t.reshape(-1, *t.shape[2:])
    for s, h in units:
        a, b = cu[s], cu[s + 1]
        pick = lambda t: flat(t)[a:b, h:h + 1].double().numpy()
        ro, rhT, _ = oracle.forward(pick(x["q"]), pick(x["k"]), pick(x["v"]), pick(x["g"]),
                                    flat(x["beta"])[a:b, h:h + 1].double().numpy(),
                                    x["A_log"][h:h + 1].double().numpy(),
                                    x["h0"][s:s + 1, h:h + 1].double().numpy(),
                                    cu_seqlens=[0, b - a])
        got = flat(o)[a:b, h].double().cpu().numpy()
        assert rel_l2(got, ro[:, 0]) <= TOL, (name, s, h)
        assert rel_l2(hT[s, h].double().cpu().numpy(), rhT[0, 0]) <= TOL, (name, s, h)
    assert torch.isfinite(o.float()).all()
