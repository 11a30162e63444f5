"""GPU parity of the context-parallel state scans.  With few (sequence, head)
chains, the library splits each sequence's chunks into P segments: every
segment is scanned locally, the inner segments' transfer matrices P_g are
formed, the segment boundaries are chained, and the segments are scanned
again from the true boundaries.  These shapes take that path (fixed length,
bf16, K = V = 128, B*H small, at least 4P chunks); KDA_SCAN_CP=n picks n
segments, KDA_SCAN_CP=0 the whole-sequence chains.  Tolerances as for the
other bf16 parity tests: 2e-2 per-tensor relative L2 against the oracle."""
import numpy as np
import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda
import oracle
from linear_attention_backward_gb300 import workloads as wl
from kda_testutil import (GRADS, check_dalog_biased, f64_tokens, gpu_bwd, oracle_bwd, oracle_states, rel_l2,
                          slot_index, to_dev, unpack_core_tiles)

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _compare(g, ref, keys=GRADS, tol=TOL):
    errs = {k: rel_l2(g[k].double().cpu().numpy().reshape(ref[k].shape), ref[k]) for k in keys}
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"rel-L2 above {tol}: {bad} (all: {errs})"
    return errs


def _tiles(ws, off, n):
    return unpack_core_tiles(ws[off:off + 2 * n].view(torch.bfloat16).reshape(-1, 128, 128))


@pytest.mark.parametrize("segs", [None, "3"])
def test_cp_backward_and_every_chunk_state(monkeypatch, segs):
    # 17 chunks with a ragged last one: 4 segments by default (4, 4, 4, 5 chunks)
    if segs is not None:
        monkeypatch.setenv("KDA_SCAN_CP", segs)
    w = wl.custom("cp", B=1, T=64 * 16 + 37, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=31)
    g, d = gpu_bwd(x)
    assert kda.get_device_status() == 0
    ref = oracle_bwd(x, want_chunk_dstates=True)
    _compare(g, ref)
    # every chunk's published state and state gradient, from each segment's
    # chain (first/last segments in phase 1, the others in phase 3)
    shape = kda.make_shape(d["q"], d["v"])
    n = kda.num_chunk_slots(shape) * 2 * 128 * 128
    ws = g["_workspace"]
    slots = np.concatenate(slot_index(x))
    cs, _ = oracle_states(x)
    st = _tiles(ws, 0, n).reshape(-1, 2, 128, 128).double().cpu().numpy()[slots]
    for c in range(len(slots)):
        assert rel_l2(st[c], cs[c]) < 1e-2, ("state", c)
    off = kda.workspace_dstates_offset(shape)
    dst = _tiles(ws, off, n).reshape(-1, 2, 128, 128).double().cpu().numpy()[slots]
    for c in range(len(slots)):
        assert rel_l2(dst[c], ref["chunk_dstates"][c]) < 1e-2, ("dstate", c)


def test_cp_matches_whole_sequence_chains(monkeypatch):
    w = wl.custom("cp", B=2, T=64 * 24, H=3, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=32)
    g_cp, _ = gpu_bwd(x)
    monkeypatch.setenv("KDA_SCAN_CP", "0")
    g_one, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    for k in GRADS:
        assert rel_l2(g_cp[k].double().cpu().numpy(), g_one[k].double().cpu().numpy()) < 1e-2, k
    _compare(g_cp, oracle_bwd(x))


def test_cp_two_chains_per_sm(monkeypatch):
    # 32 sequence-heads: three segments would need 160 first-pass chains, more
    # than one per SM, so the split takes two per SM: 4 segments, 256 chains
    w = wl.custom("cp", B=1, T=64 * 16 + 37, H=32, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=38)
    d = to_dev(x)
    assert kda.scan_segments(kda.make_shape(d["q"], d["v"])) == 4
    g_cp, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    _compare(g_cp, oracle_bwd(x))
    monkeypatch.setenv("KDA_SCAN_CP", "0")
    g_one, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    for k in GRADS:
        assert rel_l2(g_cp[k].double().cpu().numpy(), g_one[k].double().cpu().numpy()) < 1e-2, k


def test_cp_fwd_states_two_chains_per_sm_match_the_backward():
    # kda_fwd_states at the two-per-SM split (32 sequence-heads, 4 segments),
    # with the prep kernel writing the scans' operands only: its packed states
    # match the ones kda_bwd recomputes (the same scans on the full prep
    # kernel's operands) and the oracle's
    w = wl.custom("cp", B=1, T=64 * 16 + 37, H=32, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=39)
    d = to_dev(x)
    shape = kda.make_shape(d["q"], d["v"])
    assert kda.scan_segments(shape) == 4
    states, hT = kda.fwd_states(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                                want_hT=True)
    torch.cuda.synchronize()
    assert kda.get_device_status() == 0
    g, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    n = kda.num_chunk_slots(shape) * 32 * 128 * 128  # elements
    internal = g["_workspace"][:2 * n].view(torch.bfloat16)
    assert rel_l2(states.reshape(-1).double().cpu().numpy(),
                  internal.double().cpu().numpy()) < 1e-3
    cs, hT_ref = oracle_states(x)
    slots = np.concatenate(slot_index(x))
    got = unpack_core_tiles(states).double().cpu().numpy()[slots]
    assert rel_l2(got, cs) < 1e-2
    assert rel_l2(hT.double().cpu().numpy(), hT_ref) < 1e-2


def test_cp_long_segments_eight_way():
    # 128 chunks, 2 chains: 8 segments of 16 chunks and 6 combine steps
    w = wl.custom("cp", B=1, T=8192, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=33)
    g, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    _compare(g, oracle_bwd(x))


def test_cp_reverse_only_with_given_states():
    # the caller's states: only the reverse scan runs, context-parallel; its
    # dS chains are those of the full call, so the gradients agree bit for bit
    w = wl.custom("cp", B=1, T=64 * 20, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=34)
    g1, d = gpu_bwd(x)
    shape = kda.make_shape(d["q"], d["v"])
    n = kda.num_chunk_slots(shape) * 2 * 128 * 128
    internal = g1["_workspace"][:2 * n].view(torch.bfloat16).reshape(-1, 2, 128, 128)
    g2, _ = gpu_bwd(x, states=internal)
    assert kda.get_device_status() == 0
    for k in GRADS:
        assert torch.equal(g1[k], g2[k]), k


def test_cp_gate_bias():
    w = wl.custom("cp", B=1, T=64 * 16, H=2, K=128, V=128, dtype="bf16", with_h0=True,
                  with_dhT=True)
    x = wl.make_inputs(w, seed=35)
    gen = torch.Generator().manual_seed(7)
    x["dt_bias"] = torch.randn(2, 128, generator=gen) * 0.5
    g, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    ref = oracle_bwd(x)
    _compare(g, ref, keys=("dq", "dk", "dv", "dg", "dbeta", "dh0", "ddt_bias"))
    check_dalog_biased(g, ref, x, TOL)  # weaker bound: gate-bias test only


@pytest.mark.parametrize("segs", [None, "3"])
def test_cp_forward(monkeypatch, segs):
    if segs is not None:
        monkeypatch.setenv("KDA_SCAN_CP", segs)
    w = wl.custom("cpf", B=1, T=64 * 18 + 5, H=3, K=128, V=128, dtype="bf16", with_h0=True)
    x = wl.make_inputs(w, seed=36)
    d = to_dev(x)
    o, hT = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                    want_hT=True)
    torch.cuda.synchronize()
    assert kda.get_device_status() == 0
    ro, rhT, _ = oracle.forward(
        f64_tokens(x["q"]), f64_tokens(x["k"]), f64_tokens(x["v"]), f64_tokens(x["g"]),
        f64_tokens(x["beta"]), x["A_log"].double().numpy(), x["h0"].double().numpy(),
        cu_seqlens=wl.seq_bounds(x))
    assert rel_l2(o.double().cpu().numpy().reshape(ro.shape), ro) <= TOL
    assert rel_l2(hT.double().cpu().numpy(), rhT) <= TOL


def test_cp_varlen_with_short_and_empty_sequences():
    # 86 chunks over 5 sequences: 4 segments of each sequence's own chunks;
    # the empty and the 70-token sequence get empty or one-chunk segments
    lengths = [2000, 0, 1537, 70, 1900]
    w = wl.custom("cpv", H=2, K=128, V=128, dtype="bf16", with_h0=True, with_dhT=True,
                  varlen=(5, 0, 2048))
    x = wl.make_inputs(w, seed=37, lengths=lengths)
    d = to_dev(x)
    assert kda.scan_segments(kda.make_shape(d["q"], d["v"], cu_seqlens=d["cu_seqlens"])) == 4
    g, _ = gpu_bwd(x)
    assert kda.get_device_status() == 0
    ref = oracle_bwd(x)
    _compare(g, ref)
    # the same states handed back: the reverse scan alone runs, context-parallel
    # over the same segments, and reproduces every gradient bit for bit
    shape = kda.make_shape(d["q"], d["v"], cu_seqlens=d["cu_seqlens"])
    n = kda.num_chunk_slots(shape) * 2 * 128 * 128
    internal = g["_workspace"][:2 * n].view(torch.bfloat16).reshape(-1, 2, 128, 128)
    g2, _ = gpu_bwd(x, states=internal)
    assert kda.get_device_status() == 0
    for k in GRADS:
        assert torch.equal(g[k], g2[k]), k
    # the empty sequence passes its state gradient straight through (its
    # boundaries cross the tf32 combine: identity products rounded to 2^-11)
    np.testing.assert_allclose(g["dh0"][1].cpu().numpy(), x["dhT"][1].numpy(), rtol=1e-3,
                               atol=1e-6)
    # the forward pass on the same batch
    o, hT = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                    cu_seqlens=d["cu_seqlens"], want_hT=True)
    torch.cuda.synchronize()
    assert kda.get_device_status() == 0
    ro, rhT, _ = oracle.forward(
        f64_tokens(x["q"]), f64_tokens(x["k"]), f64_tokens(x["v"]), f64_tokens(x["g"]),
        f64_tokens(x["beta"]), x["A_log"].double().numpy(), x["h0"].double().numpy(),
        cu_seqlens=wl.seq_bounds(x))
    assert rel_l2(o.double().cpu().numpy().reshape(ro.shape), ro) <= TOL
    assert rel_l2(hT.double().cpu().numpy(), rhT) <= TOL
    np.testing.assert_allclose(hT[1].cpu().numpy(), x["h0"][1].numpy(), rtol=1e-3, atol=1e-6)
