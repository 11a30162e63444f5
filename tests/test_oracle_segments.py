"""Pin of the segment algebra the context-parallel scans rely on, from the
token-serial oracle alone.  Over a segment of tokens [a, b) the state update
is affine in the state: S_b = P S_a + E, with P the segment's transfer (its
forward with v = 0 started from the identity) and E its forward from zero;
and the adjoint is affine in the end gradient: dS_a = P^T dS_b + F, with F
the segment's dh0 for dh_T = 0.  The segment boundaries, the full sequence's
chunk states and its chunk state gradients all come from the oracle; fp64."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("seg", [(1, 4), (0, 2), (2, 5)])
def test_segment_transfer_composes_states_and_state_gradients(seg):
    rng = np.random.default_rng(sum(seg))
    C, nck, H, K = 16, 5, 2, 4          # K = V: the transfer is a K x K matrix
    T = C * nck
    q, k, v, g = (rng.standard_normal((T, H, K)) for _ in range(4))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    A_log = rng.uniform(0, 1.5, (H,))
    h0 = 0.3 * rng.standard_normal((1, H, K, K))
    dO = rng.standard_normal((T, H, K))
    dhT = rng.standard_normal((1, H, K, K))
    cu = [0, T]
    _, _, states = oracle.forward(q, k, v, g, beta, A_log, h0, cu_seqlens=cu, chunk=C,
                                  want_chunk_states=True)
    full = oracle.backward(q, k, v, g, beta, A_log, h0, dO, dhT, cu_seqlens=cu, chunk=C,
                           want_chunk_dstates=True)
    ca, cb = seg
    a, b = C * ca, C * cb
    sl = slice(a, b)
    L = [0, b - a]
    zero = np.zeros((1, H, K, K))
    eye = np.broadcast_to(np.eye(K), (1, H, K, K)).copy()
    _, E, _ = oracle.forward(q[sl], k[sl], v[sl], g[sl], beta[sl], A_log, zero, cu_seqlens=L,
                             chunk=C)
    _, P, _ = oracle.forward(q[sl], k[sl], np.zeros_like(v[sl]), g[sl], beta[sl], A_log, eye,
                             cu_seqlens=L, chunk=C)
    S_a = states[ca]
    _, hT_full, _ = oracle.forward(q, k, v, g, beta, A_log, h0, cu_seqlens=cu, chunk=C)
    S_b = states[cb] if cb < nck else hT_full[0]
    np.testing.assert_allclose(np.einsum("hck,hkv->hcv", P[0], S_a) + E[0], S_b,
                               rtol=1e-10, atol=1e-12)
    # reverse: dS at the segment's start and end from the full backward
    # (chunk_dstates[n] is the gradient of the state at the end of chunk n)
    dS_a = full["chunk_dstates"][ca - 1] if ca > 0 else full["dh0"][0]
    dS_b = full["chunk_dstates"][cb - 1]
    F = oracle.backward(q[sl], k[sl], v[sl], g[sl], beta[sl], A_log, zero, dO[sl], zero,
                        cu_seqlens=L, chunk=C)["dh0"][0]
    np.testing.assert_allclose(np.einsum("hkc,hkv->hcv", P[0], dS_b) + F, dS_a,
                               rtol=1e-10, atol=1e-12)
