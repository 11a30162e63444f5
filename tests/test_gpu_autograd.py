"""The autograd layer (KDAFunction: kda_fwd forward, kda_bwd backward) on the
GPU: its gradients are those of a direct kda_bwd call, bit for bit, for the
loss <dO, o> + <dh_T, hT>; the forward's o matches kda_fwd."""
import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda
from linear_attention_backward_gb300 import workloads as wl
from kda_testutil import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("varlen", [False, True])
def test_autograd_matches_direct_backward(varlen):
    if varlen:
        w = wl.custom("ag", H=2, K=128, V=128, dtype="bf16", with_h0=True, with_dhT=True,
                      varlen=(3, 1, 200))
        x = wl.make_inputs(w, seed=51, lengths=[130, 0, 77])
    else:
        w = wl.custom("ag", B=2, T=150, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                      with_dhT=True)
        x = wl.make_inputs(w, seed=51)
    d = to_dev(x)
    d["dt_bias"] = (0.3 * torch.randn(2, 128, generator=torch.Generator().manual_seed(2))).cuda()
    leaves = {n: d[n].clone().requires_grad_(True)
              for n in ("q", "k", "v", "g", "beta", "A_log", "h0", "dt_bias")}
    o, hT = kda.kda(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                    leaves["A_log"], leaves["h0"], dt_bias=leaves["dt_bias"],
                    cu_seqlens=d["cu_seqlens"])
    o_ref, hT_ref = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                            cu_seqlens=d["cu_seqlens"], want_hT=True, dt_bias=d["dt_bias"])
    assert torch.equal(o, o_ref) and torch.equal(hT, hT_ref)
    loss = (o.float() * d["dO"].float()).sum() + (hT * d["dhT"]).sum()
    loss.backward()
    ref = kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"], d["dO"],
                  d["dhT"], cu_seqlens=d["cu_seqlens"], dt_bias=d["dt_bias"])
    torch.cuda.synchronize()
    assert kda.get_device_status() == 0
    pairs = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "A_log": "dA_log",
             "h0": "dh0", "dt_bias": "ddt_bias"}
    for leaf, key in pairs.items():
        assert torch.equal(leaves[leaf].grad, ref[key]), leaf
