"""The C-ABI library loads on a machine without a GPU, exports every entry
point include/kda.h declares, and validates arguments on the host (these
calls return before anything touches CUDA)."""
import ctypes
import os
import re

import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return kda.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert {"kda_bwd", "kda_fwd", "kda_fwd_states", "kda_workspace_bytes"} <= names
    for n in sorted(names):
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_abi_version_and_strings(L):
    assert L.kda_abi_version() == 7
    for st in range(9):
        assert len(L.kda_status_str(st)) > 0


def _shape(**kw):
    d = dict(B=2, T=130, H=3, K=128, V=128, chunk=64, num_seqs=0, cu_seqlens=None,
             scale=0.0, l2_eps=-1.0, dtype=kda.KDA_BF16)
    d.update(kw)
    return kda.KdaShape(d["B"], d["T"], d["H"], d["K"], d["V"], d["chunk"], d["num_seqs"],
                        d["cu_seqlens"], d["scale"], d["l2_eps"], d["dtype"])


def test_slots_and_workspace(L):
    s = _shape()
    assert kda.num_chunk_slots(s) == 2 * 3
    sb = 6 * 3 * 128 * 128 * 2
    sb = (sb + 255) // 256 * 256
    assert kda.workspace_dstates_offset(s) == sb
    # states, dS, dA_log and ddt_bias partials and (bf16, K = V = 128) the
    # per-chunk operand blocks of the tcgen05 path, 107008 bytes per (slot,
    # head), and its range flags, 4 bytes per (slot, head)
    prep = (6 * 3 * 107008 + 255) // 256 * 256
    ddt = (6 * 3 * 128 * 4 + 255) // 256 * 256
    flags = (6 * 3 * 4 + 255) // 256 * 256
    assert kda.workspace_bytes(s) == (2 * sb + ((6 * 3 * 4 + 255) // 256) * 256 + ddt + prep
                                      + flags)
    v = _shape(B=1, T=300, num_seqs=4, cu_seqlens=0x1000)
    assert kda.num_chunk_slots(v) == 300 // 64 + 4
    assert kda.scan_segments(v) == 0 and kda.scan_segments(s) == 0
    # varlen: P from the average chunks per sequence (86 chunks / 5 sequences)
    v = _shape(B=1, T=5507, num_seqs=5, cu_seqlens=0x1000)
    assert kda.scan_segments(v) == 4
    r = lambda x: (x + 255) // 256 * 256
    n = (5507 // 64 + 5) * 3
    assert kda.workspace_bytes(v) == (2 * r(n * 128 * 128 * 2) + r(n * 4) + r(n * 128 * 4)
                                      + r(n * 107008) + r(5 * 3 * 8 * 128 * 128 * 4)
                                      + r(n * 4))
    f = _shape(K=64, V=64, dtype=kda.KDA_FP32, T=64, B=1)
    assert kda.workspace_dstates_offset(f) == 1 * 3 * 64 * 64 * 4
    sf = 1 * 3 * 64 * 64 * 4
    # no operand blocks off the tcgen05 path
    assert kda.workspace_bytes(f) == 2 * sf + 256 + 3 * 64 * 4
    # few (sequence, head) chains and 16 chunks: the context-parallel scans take
    # P = 4 segments of 4 chunks and 3P - 4 = 8 fp32 boundary tiles per
    # (sequence, head) at the end of the workspace
    r = lambda x: (x + 255) // 256 * 256
    c = _shape(B=1, T=1024)
    assert kda.scan_segments(c) == 4
    n = 16 * 3
    base = 2 * r(n * 128 * 128 * 2) + r(n * 4) + r(n * 128 * 4) + r(n * 107008)
    assert kda.workspace_bytes(c) == base + r(3 * 8 * 128 * 128 * 4) + r(n * 4)
    # 15 chunks allow 3 segments (5 tiles); varlen shapes use whole-sequence chains
    c = _shape(B=1, T=960)
    assert kda.scan_segments(c) == 3
    n = 15 * 3
    base = 2 * r(n * 128 * 128 * 2) + r(n * 4) + r(n * 128 * 4) + r(n * 107008)
    assert kda.workspace_bytes(c) == base + r(3 * 5 * 128 * 128 * 4) + r(n * 4)


def test_pad64_workspace_layout(L):
    # bf16 K = V = 64 runs on zero-padded 128-channel copies: the workspace is
    # the 128-channel shape's own (states, dS, partials, operand blocks, range
    # flags), then the padded q, k, v, g, dO and dq, dk, dv, dg, h0 / dh_T / dh0
    # tiles, the gate bias and its gradient, and the padded given states
    r = lambda x: (x + 255) // 256 * 256
    B, T, H = 2, 150, 3
    s = _shape(B=B, T=T, H=H, K=64, V=64)
    slots = B * ((T + 63) // 64)
    n = slots * H
    assert kda.scan_segments(s) == 0  # 3 chunks per sequence: too few to split
    inner = r(2 * r(n * 128 * 128 * 2) + r(n * 4) + r(n * 128 * 4) + r(n * 107008) + r(n * 4))
    pads = (9 * r(B * T * H * 128 * 2) + 3 * r(B * H * 128 * 128 * 4) + 2 * r(H * 128 * 4)
            + r(n * 128 * 128 * 2))
    assert kda.workspace_bytes(s) == inner + pads
    # the state gradients sit after the padded shape's states
    assert kda.workspace_dstates_offset(s) == r(n * 128 * 128 * 2)


@pytest.mark.parametrize("kw,code", [
    (dict(K=96, V=96), 2), (dict(K=128, V=64), 2), (dict(chunk=32), 2),
    (dict(B=0), 1), (dict(H=0), 1), (dict(T=-1), 1), (dict(dtype=7), 1),
    (dict(num_seqs=3), 1), (dict(cu_seqlens=0x1000, num_seqs=2), 1),
    (dict(K=128, V=128, dtype=kda.KDA_FP32), 2),
])
def test_bad_shapes_rejected(L, kw, code):
    s = _shape(**kw)
    assert kda.workspace_bytes(s) == 0
    fake = ctypes.c_void_p(1 << 20)
    st = L.kda_bwd(ctypes.byref(s), *([fake] * 19), fake, ctypes.c_size_t(1 << 40), None)
    assert st == code


def test_bwd_pointer_checks(L):
    s = _shape()
    fake = ctypes.c_void_p(1 << 20)
    args = [fake] * 19
    ws_ok = ctypes.c_size_t(kda.workspace_bytes(s))
    # a required pointer missing
    a = list(args); a[0] = None
    assert L.kda_bwd(ctypes.byref(s), *a, fake, ws_ok, None) == 1
    # misaligned tensor
    a = list(args); a[3] = ctypes.c_void_p((1 << 20) + 4)
    assert L.kda_bwd(ctypes.byref(s), *a, fake, ws_ok, None) == 1
    # workspace: missing, too small, misaligned
    assert L.kda_bwd(ctypes.byref(s), *args, None, ws_ok, None) == 3
    assert L.kda_bwd(ctypes.byref(s), *args, fake, ctypes.c_size_t(ws_ok.value - 1), None) == 3
    assert L.kda_bwd(ctypes.byref(s), *args, ctypes.c_void_p((1 << 20) + 16), ws_ok, None) == 3
    # fwd_states: missing states; missing q (the tcgen05 path's prep needs it);
    # workspace missing or too small
    a = [fake] * 6 + [None, None, fake, None]  # q k v g beta A_log, dt_bias, h0, states, hT
    b = list(a); b[8] = None
    assert L.kda_fwd_states(ctypes.byref(s), *b, fake, ws_ok, None) == 1
    b = list(a); b[0] = None
    assert L.kda_fwd_states(ctypes.byref(s), *b, fake, ws_ok, None) == 1
    assert L.kda_fwd_states(ctypes.byref(s), *a, None, ws_ok, None) == 3
    assert L.kda_fwd_states(ctypes.byref(s), *a, fake, ctypes.c_size_t(ws_ok.value - 1),
                            None) == 3
    # the selftest's layouts are 0 (packed), 1 (padded) and 2 (128-byte
    # swizzled, K in slabs of 64) only
    assert L.kda_selftest_umma(fake, fake, fake, 64, 64, 0, 0, 3, None) == 1
    assert L.kda_selftest_umma(fake, fake, fake, 64, 32, 0, 0, 2, None) == 1


def test_host_cu_seqlens_check(L):
    good = torch.tensor([0, 5, 5, 70], dtype=torch.int32)
    assert kda.check_cu_seqlens_host(good, 70) == 0
    assert kda.check_cu_seqlens_host(good, 71) == 1
    assert kda.check_cu_seqlens_host(torch.tensor([1, 5, 70], dtype=torch.int32), 70) == 1
    assert kda.check_cu_seqlens_host(torch.tensor([0, 9, 5, 70], dtype=torch.int32), 70) == 1


def test_fwd_argument_checks(L):
    s = _shape()
    fake = ctypes.c_void_p(1 << 20)
    ws_ok = ctypes.c_size_t(kda.workspace_bytes(s))
    args = [fake] * 6 + [None, None, fake, None]  # q k v g beta A_log, dt_bias, h0, o, hT
    # a required pointer missing, a misaligned one
    a = list(args); a[8] = None
    assert L.kda_fwd(ctypes.byref(s), *a, fake, ws_ok, None) == 1
    a = list(args); a[2] = ctypes.c_void_p((1 << 20) + 2)
    assert L.kda_fwd(ctypes.byref(s), *a, fake, ws_ok, None) == 1
    # workspace missing or too small
    assert L.kda_fwd(ctypes.byref(s), *args, None, ws_ok, None) == 3
    assert L.kda_fwd(ctypes.byref(s), *args, fake, ctypes.c_size_t(ws_ok.value - 1), None) == 3
    # the forward runs bf16 only (K = V = 64 on zero-padded copies): fp32 is
    # not built
    f = _shape(dtype=kda.KDA_FP32, K=64, V=64)
    assert L.kda_fwd(ctypes.byref(f), *args, fake, ctypes.c_size_t(1 << 40), None) == 2


@pytest.mark.parametrize("B,T,H,expect", [
    (1, 4096, 16, 4),     # 16 sequence-heads: (3P - 4) * 16 <= 152 -> P = 4
    (1, 8192, 2, 8),      # 2 sequence-heads, 128 chunks: capped at 8
    (1, 1024, 2, 4),      # 16 chunks: at least 4 per segment -> P = 4
    (1, 704, 2, 0),       # 11 chunks: fewer than 4 per segment for P = 3
    (4, 8192, 19, 0),     # 2 * 76 chains fill the 152 SMs
    (1, 8192, 30, 3),     # 30: (3 * 3 - 4) * 30 = 150 <= 152
    (1, 8192, 32, 4),     # 32: (3 * 3 - 4) * 32 > 152, so two per SM: 8 * 32 = 256 <= 304
    (1, 8192, 38, 4),     # 38: two per SM, (3 * 4 - 4) * 38 = 304 <= 304 -> P = 4
    (1, 8192, 39, 0),     # 39: the whole-sequence chains fill more than half the SMs
    (1, 768, 32, 3),      # two per SM, 12 chunks: at least 4 per segment -> P = 3
])
def test_scan_segments_rule(L, B, T, H, expect):
    assert kda.scan_segments(_shape(B=B, T=T, H=H)) == expect
    # bf16 K = V = 64 runs the same scans on zero-padded copies; fp32 runs
    # the per-band scans: no segments
    assert kda.scan_segments(_shape(B=B, T=T, H=H, K=64, V=64)) == expect
    assert kda.scan_segments(_shape(B=B, T=T, H=H, K=64, V=64, dtype=kda.KDA_FP32)) == 0


@pytest.mark.parametrize("env,expect", [("0", 0), ("3", 3), ("4", 4), ("9", 4), ("2", 4),
                                        ("x", 0)])
def test_scan_segments_env_override(L, monkeypatch, env, expect):
    # KDA_SCAN_CP=0 (or anything non-numeric) turns the split off; 3..P takes
    # that many segments; other values keep the shape's own P (4 here)
    monkeypatch.setenv("KDA_SCAN_CP", env)
    assert kda.scan_segments(_shape(B=1, T=4096, H=16)) == expect
