"""Host-side logic without a GPU: the binding fails loudly when the CUDA
library is missing (there is no fallback path), and bench.py's per-workload
decisions (which workloads flush L2 between timed steps, how many kernels
one call launches) follow the library's own report."""
import importlib.util
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_binding_raises_without_the_library(tmp_path):
    # a fresh interpreter whose binding points at a library that does not exist
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import linear_attention_backward_gb300 as kda\n"
        "kda._LIB_PATH = %r\n"
        "kda._lib = None\n"
        "try:\n"
        "    kda.lib()\n"
        "except ImportError as e:\n"
        "    print('raised', 'not built' in str(e))\n"
        "else:\n"
        "    print('loaded')\n" % (ROOT, str(tmp_path / "absent" / "libkda.so")))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=300)
    assert out.stdout.strip() == "raised True", out.stdout + out.stderr


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_bench_flushes_l2_only_for_small_inputs():
    b = _bench()
    from linear_attention_backward_gb300 import workloads as wl
    assert b.flushes_l2(wl.WORKLOADS["lowpar_bf16"])      # 17 MB per input tensor
    assert b.flushes_l2(wl.WORKLOADS["tiny_fp32"])
    assert not b.flushes_l2(wl.WORKLOADS["main_bf16"])    # 268 MB per input tensor
    assert not b.flushes_l2(wl.WORKLOADS["large_bf16"])
    assert not b.flushes_l2(wl.WORKLOADS["varlen_bf16"])


@pytest.mark.parametrize("name,bwd,fwd", [("main_bf16", 6, 4), ("lowpar_bf16", 8, 6),
                                          ("varlen_bf16", 7, 5), ("tiny_fp32", 4, 3)])
def test_bench_counts_the_launches_of_one_call(name, bwd, fwd):
    # prep, scans, gradients, reduction; varlen adds the sequence order; the
    # context-parallel scans (low parallelism) add the combine and a second
    # pass; bf16 K = V = 128 adds the exact range kernels (two in the
    # backward, one in the forward)
    b = _bench()
    import torch
    import linear_attention_backward_gb300 as kda
    from linear_attention_backward_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    cu = None
    if w.varlen:
        # the recipe's first draw: the sequence lengths (seed 0)
        n, lo, hi = w.varlen
        T = int(torch.randint(lo, hi + 1, (n,), generator=torch.Generator().manual_seed(0)).sum())
        q = torch.empty((1, T, w.H, w.K), dtype=torch.bfloat16, device="meta")
        cu = torch.empty(w.varlen[0] + 1, dtype=torch.int32, device="meta")
    else:
        q = torch.empty((w.B, w.T, w.H, w.K), dtype=torch.bfloat16, device="meta")
    shape = kda.make_shape(q, q, cu_seqlens=cu)
    if cu is not None:
        shape.cu_seqlens = 0x1000  # a non-null pointer: the host never reads it
    assert b.launches_per_step(shape, cu) == bwd
    assert b.launches_per_step(shape, cu, forward=True) == fwd
