"""Bounded device-side waits, exercised without a fault.

Every wait of a kernel on a copy or a tensor-core product polls a bounded
number of times; a CTA whose wait gives up records KDA_ERR_TIMEOUT (5) in the
device status word, issues no further product, writes no further result,
drains what it has in flight and releases its Tensor Memory.  The test hook
KDA_TEST_STARVE_WAITS makes the named kernel arm its first load barrier
without issuing the copies that would complete it (a barrier nothing
completes) and caps the call's waits at 4096 polls.  The call must report
the timeout, and the next call on the same context must be clean and match
the oracle."""
import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda
from linear_attention_backward_gb300 import workloads as wl
from kda_testutil import GRADS, gpu_bwd, oracle_bwd, rel_l2, to_dev

pytestmark = pytest.mark.gpu

KDA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("kernel", ["prep", "scan", "grads", "out"])
def test_starved_wait_reports_timeout_and_the_next_call_is_clean(monkeypatch, kernel):
    w = wl.custom("to", B=1, T=100, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=61)
    d = to_dev(x)
    assert kda.get_device_status() == 0
    monkeypatch.setenv("KDA_TEST_STARVE_WAITS", kernel)
    if kernel == "out":  # the forward's output kernel
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"])
    else:
        kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"], d["dO"],
                d["dhT"])
    assert kda.get_device_status() == KDA_ERR_TIMEOUT
    monkeypatch.delenv("KDA_TEST_STARVE_WAITS")
    # the context stays usable: the same call again is clean and right
    g, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    ref = oracle_bwd(x)
    for key in GRADS:
        got = g[key].double().cpu().numpy().reshape(ref[key].shape)
        assert rel_l2(got, ref[key]) <= 2e-2, key
