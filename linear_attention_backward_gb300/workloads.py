"""Seeded synthetic workloads for the KDA backward pass.

This module holds only input recipes (shapes, distributions, seeds).  It has
none of the method's arithmetic, so both the CUDA path's tests/benchmark and
the CPU oracle can draw their inputs from it.

Recipe (all configurations): one CPU ``torch.Generator`` seeded with ``seed``
draws, in this fixed order, the varlen lengths (varlen only), q, k, v, g,
beta_raw, A_log, dO, h0, dh_T.  q, k, v, dO, g ~ N(0, 1) (q and k raw: the
library L2-normalises them), beta = sigmoid(N(0, 1)), A_log ~ U(0, 1.5) per
head, h0 ~ N(0, 0.1^2) and dh_T ~ N(0, 1) where the configuration has them
(else zero).  Tensors are then cast to the configuration's dtype; A_log, h0
and dh_T stay fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: str                     # "fp32" or "bf16"
    with_h0: bool = False
    with_dhT: bool = False
    varlen: tuple = field(default=())  # (num_seqs, lo, hi) for U[lo, hi] lengths
    chunk: int = 64

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16


WORKLOADS = {
    # B=1 T=256 H=2 K=V=64, fp32 inputs
    "tiny_fp32": Workload("tiny_fp32", 1, 256, 2, 64, 64, "fp32"),
    # B=1 T=4096 H=16 K=V=128, bf16 (low parallelism: 16 sequence-heads)
    "lowpar_bf16": Workload("lowpar_bf16", 1, 4096, 16, 128, 128, "bf16"),
    # B=4 T=8192 H=32 K=V=128, bf16 (the main benchmark workload)
    "main_bf16": Workload("main_bf16", 4, 8192, 32, 128, 128, "bf16"),
    # a quarter of the main batch (B=1), the size used for ncu captures
    "main_b1_bf16": Workload("main_b1_bf16", 1, 8192, 32, 128, 128, "bf16"),
    # B=8 T=16384 H=32 K=V=128, bf16, with h0 and dh_T
    "large_bf16": Workload("large_bf16", 8, 16384, 32, 128, 128, "bf16", True, True),
    # 16 packed sequences, lengths U[512, 8192], H=32 K=V=128, bf16, h0 and dh_T
    "varlen_bf16": Workload("varlen_bf16", 1, 0, 32, 128, 128, "bf16", True, True,
                            varlen=(16, 512, 8192)),
}


def custom(name="custom", B=1, T=64, H=2, K=128, V=128, dtype="bf16",
           with_h0=False, with_dhT=False, varlen=()):
    """A workload of any shape with the same distributions."""
    return Workload(name, B, T, H, K, V, dtype, with_h0, with_dhT, tuple(varlen))


def make_inputs(w: Workload, seed: int = 0, lengths=None):
    """Draw the inputs of workload ``w`` on the host.

    Returns a dict of CPU tensors: q, k, g [B, T, H, K]; v, dO [B, T, H, V];
    beta [B, T, H] (dtype of ``w``); A_log [H]; h0, dhT [N, H, K, V] (fp32,
    zeros when the workload has none); cu_seqlens (int32 [N + 1], or None for
    fixed-length batches).  Varlen workloads are packed as B = 1.
    ``lengths`` overrides the drawn varlen lengths.
    """
    gen = torch.Generator().manual_seed(seed)
    cu = None
    B, T = w.B, w.T
    if w.varlen:
        n, lo, hi = w.varlen
        drawn = torch.randint(lo, hi + 1, (n,), generator=gen).tolist()
        if lengths is None:
            lengths = drawn
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
        B, T = 1, int(cu[-1])
    N = len(lengths) if w.varlen else B
    H, K, V = w.H, w.K, w.V
    f32 = torch.float32

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=f32)

    q = randn(B, T, H, K)
    k = randn(B, T, H, K)
    v = randn(B, T, H, V)
    g = randn(B, T, H, K)
    beta = torch.sigmoid(randn(B, T, H))
    A_log = torch.rand(H, generator=gen, dtype=f32) * 1.5
    dO = randn(B, T, H, V)
    h0 = randn(N, H, K, V) * 0.1 if w.with_h0 else torch.zeros(N, H, K, V)
    dhT = randn(N, H, K, V) if w.with_dhT else torch.zeros(N, H, K, V)
    dt = w.torch_dtype
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), g=g.to(dt), beta=beta.to(dt),
                A_log=A_log, dO=dO.to(dt), h0=h0, dhT=dhT, cu_seqlens=cu)


def seq_bounds(inputs):
    """cu_seqlens as a python list (fixed-length batches: multiples of T)."""
    cu = inputs["cu_seqlens"]
    if cu is not None:
        return [int(x) for x in cu.tolist()]
    B, T = inputs["q"].shape[:2]
    return [b * T for b in range(B + 1)]
