"""bf16 K = V = 64 on the 128-channel tensor-core kernels (zero-padded copies).

A padded channel has q^ = k^ = 0 and zero value columns, so its state rows and
columns stay zero and every gradient term that touches it vanishes: the real
channels' results are those of the 64-channel problem (read-out scale 64^-1/2).
Parity against the fp64 oracle at the bf16 tolerance (2e-2 per-tensor relative
L2), and against the mma.sync kernels that KDA_PAD64=0 selects."""
import numpy as np
import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda
import oracle
from linear_attention_backward_gb300 import workloads as wl
from kda_testutil import GRADS, f64_tokens, gpu_bwd, oracle_bwd, rel_l2, to_dev

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _compare(g, ref, keys=GRADS):
    errs = {k: rel_l2(g[k].double().cpu().numpy().reshape(ref[k].shape), ref[k]) for k in keys}
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    assert not bad, f"rel-L2 above {TOL}: {bad} (all: {errs})"
    return errs


@pytest.mark.parametrize("T", [1, 70, 256])
def test_pad64_backward_matches_oracle_and_mma_sync(monkeypatch, T):
    w = wl.custom("p64", B=2, T=T, H=3, K=64, V=64, dtype="bf16", with_h0=True, with_dhT=True)
    x = wl.make_inputs(w, seed=90 + T)
    ref = oracle_bwd(x)
    g, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    _compare(g, ref)
    monkeypatch.setenv("KDA_PAD64", "0")  # the mma.sync kernels
    g2, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    _compare(g2, ref)


def test_pad64_varlen_with_bias_and_given_states():
    lengths = [130, 0, 64, 5, 200]
    w = wl.custom("p64v", H=2, K=64, V=64, dtype="bf16", with_h0=True, with_dhT=True,
                  varlen=(5, 0, 256))
    x = wl.make_inputs(w, seed=93, lengths=lengths)
    gen = torch.Generator().manual_seed(94)
    x["dt_bias"] = torch.randn(2, 64, generator=gen) * 0.5
    ref = oracle_bwd(x)
    g, d = gpu_bwd(x)
    assert kda.get_device_status() == 0
    keys = tuple(k for k in GRADS if k != "dA_log") + ("ddt_bias",)
    _compare(g, ref, keys)
    # the states from kda_fwd_states (row-major 64 x 64 for this shape) handed
    # to kda_bwd, which packs them into the padded layout
    states = kda.fwd_states(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                            cu_seqlens=d["cu_seqlens"], dt_bias=d["dt_bias"])
    g2, _ = gpu_bwd(x, states=states)
    assert kda.get_device_status() == 0
    _compare(g2, ref, keys)


def test_pad64_forward():
    w = wl.custom("p64f", B=2, T=150, H=2, K=64, V=64, dtype="bf16", with_h0=True)
    x = wl.make_inputs(w, seed=95)
    d = to_dev(x)
    o, hT = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                    want_hT=True)
    torch.cuda.synchronize()
    assert kda.get_device_status() == 0
    ro, rhT, _ = oracle.forward(
        f64_tokens(x["q"]), f64_tokens(x["k"]), f64_tokens(x["v"]), f64_tokens(x["g"]),
        f64_tokens(x["beta"]), x["A_log"].double().numpy(), x["h0"].double().numpy(),
        cu_seqlens=wl.seq_bounds(x))
    assert o.shape == (2, 150, 2, 64) and hT.shape == (2, 2, 64, 64)
    assert rel_l2(o.double().cpu().numpy().reshape(ro.shape), ro) <= TOL
    assert rel_l2(hT.double().cpu().numpy(), rhT) <= TOL
    assert np.isfinite(o.float().cpu().numpy()).all()
