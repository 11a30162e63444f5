"""kda_bwd_noalloc: the backward entry point for callers that cannot allocate
device memory (it keeps its scratch in a fixed array inside the library
instead of a caller workspace).  Its results must equal kda_bwd's bit for
bit, call after call, after a call on another problem, without reserving
device memory, and it must refuse problems larger than its fixed scratch.

This file is named to be collected last, so that a failure here leaves every
other test already run."""
import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda
from linear_attention_backward_gb300 import workloads as wl
from kda_testutil import GRADS, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _fresh_out(d, H, N, K, V):
    o = {n: torch.full_like(d[m], float("nan")) for n, m in
         (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"))}
    o["dA_log"] = torch.full((H,), float("nan"), dtype=torch.float32, device="cuda")
    o["dh0"] = torch.full((N, H, K, V), float("nan"), dtype=torch.float32, device="cuda")
    return o


def _case(case):
    if case == "fixed":
        w = wl.custom("na", B=2, T=333, H=3, K=128, V=128, dtype="bf16", with_h0=True,
                      with_dhT=True)
        return wl.make_inputs(w, seed=21)
    if case == "context-parallel":
        # few chains and 20 chunks: the scans' segment boundary tiles live in
        # the fixed scratch too
        w = wl.custom("nacp", B=1, T=64 * 20, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                      with_dhT=True)
        return wl.make_inputs(w, seed=23)
    w = wl.custom("nav", H=2, K=128, V=128, dtype="bf16", with_h0=True, with_dhT=True,
                  varlen=(4, 1, 300))
    return wl.make_inputs(w, seed=22, lengths=[130, 1, 0, 257])


def _noalloc(d, out):
    kda.bwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"], d["dO"],
                    d["dhT"], cu_seqlens=d["cu_seqlens"], out=out)


# the problem each case runs first: a different shape and different inputs,
# so that a call reading scratch left over from an earlier call instead of
# writing it first would give different gradients
_OTHER = {"fixed": "varlen", "varlen": "context-parallel", "context-parallel": "fixed"}


@pytest.mark.parametrize("case", ["fixed", "varlen", "context-parallel"])
def test_noalloc_matches_workspace_entry_point_twice(case):
    x = _case(case)
    d = to_dev(x)
    # the reference: kda_bwd with a freshly allocated workspace
    ref = kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"], d["dO"],
                  d["dhT"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    shape = kda.make_shape(d["q"], d["v"], cu_seqlens=d["cu_seqlens"])
    assert kda.workspace_bytes(shape) <= kda.noalloc_scratch_bytes()
    assert (kda.scan_segments(shape) > 0) == (case == "context-parallel")
    N, H = d["h0"].shape[:2]
    # a warm-up call on another problem (the first call on a device may load
    # the module that holds the scratch array)
    do = to_dev(_case(_OTHER[case]))
    No, Ho = do["h0"].shape[:2]
    _noalloc(do, _fresh_out(do, Ho, No, 128, 128))
    torch.cuda.synchronize()
    assert kda.get_device_status() == 0
    for call in range(2):
        out = _fresh_out(d, H, N, 128, 128)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        _noalloc(d, out)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before, call  # nothing reserved
        assert kda.get_device_status() == 0
        # the same kernels on the same inputs: bit for bit kda_bwd's results
        for key in GRADS:
            assert torch.equal(out[key], ref[key]), (call, key)


def test_noalloc_rejects_problems_beyond_its_scratch():
    cap = kda.noalloc_scratch_bytes()
    assert cap == 64 << 20
    # the main workload needs far more scratch than the fixed array holds
    big = kda.KdaShape(4, 8192, 32, 128, 128, 64, 0, None, 0.0, -1.0, kda.KDA_BF16)
    assert kda.workspace_bytes(big) > cap
    fake = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    import ctypes
    p = ctypes.c_void_p(fake.data_ptr())
    st = kda.lib().kda_bwd_noalloc(ctypes.byref(big), *([p] * 18), None)
    assert st == 7
