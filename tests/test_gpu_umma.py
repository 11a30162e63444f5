"""Device self-test of the fifth-generation tensor-core building blocks
(tcgen05 MMA from shared-memory descriptors into Tensor Memory, read back
with tcgen05.ld): D = A B^T against a plain fp32 product, for K-major and
MN-major operand tiles in the packed and padded core-matrix layouts and the
128-byte swizzled layout."""
import ctypes

import pytest
import torch

import __graft_entry__
import linear_attention_backward_gb300 as kda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N", [32, 64, 128])
@pytest.mark.parametrize("K", [16, 64, 128])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("layout", [0, 1, 2])
def test_umma_tile(N, K, a_mn, b_mn, layout):
    # layout 2, the 128-byte swizzled one, takes K in slabs of 64 and (read
    # MN-major) N in slabs of 64
    if layout == 2 and (K % 64 or (b_mn and N < 64)):
        pytest.skip("not a 128-byte swizzled shape")
    __graft_entry__.build()
    L = kda.lib()
    L.kda_selftest_umma.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    L.kda_selftest_umma.restype = ctypes.c_int
    g = torch.Generator(device="cuda").manual_seed(N * 1000 + K * 10 + 2 * a_mn + b_mn)
    A = torch.randn(128, K, device="cuda", generator=g).bfloat16()
    B = torch.randn(N, K, device="cuda", generator=g).bfloat16()
    D = torch.full((128, N), float("nan"), device="cuda")
    st = L.kda_selftest_umma(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, a_mn, b_mn, layout,
                             None)
    torch.cuda.synchronize()
    assert st == 0 and kda.get_device_status() == 0
    ref = A.float() @ B.float().T
    assert ((D - ref).norm() / ref.norm()).item() < 1e-6
