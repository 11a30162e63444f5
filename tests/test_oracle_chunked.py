"""Pin of the chunk algebra: the chunked fp64 restatement (WY inverse, masks,
reverse state-gradient scan, per-chunk gradient terms) equals the
token-serial definition for several chunk sizes, ragged tails and h0/dh_T."""
import numpy as np
import pytest

import oracle
from oracle import chunked

KEYS = ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "dh0")


def _inputs(rng, Ttot, H, K, V, N):
    return dict(
        q=rng.standard_normal((Ttot, H, K)), k=rng.standard_normal((Ttot, H, K)),
        v=rng.standard_normal((Ttot, H, V)), g=rng.standard_normal((Ttot, H, K)),
        beta=1 / (1 + np.exp(-rng.standard_normal((Ttot, H)))),
        A_log=rng.uniform(0, 1.5, (H,)), h0=0.1 * rng.standard_normal((N, H, K, V)),
        dO=rng.standard_normal((Ttot, H, V)), dhT=rng.standard_normal((N, H, K, V)))


@pytest.mark.parametrize("C", [4, 16, 64])
@pytest.mark.parametrize("cu", [[0, 130], [0, 1, 63, 128, 193]])
def test_chunked_equals_token_serial(C, cu):
    rng = np.random.default_rng(C + len(cu))
    H, K, V = 2, 8, 6
    d = _inputs(rng, cu[-1], H, K, V, len(cu) - 1)
    ref = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                          d["dO"], d["dhT"], cu_seqlens=cu, chunk=C,
                          want_chunk_dstates=True)
    got = chunked.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                           d["dO"], d["dhT"], cu_seqlens=cu, chunk=C)
    for key in KEYS:
        err = np.linalg.norm(got[key] - ref[key]) / np.linalg.norm(ref[key])
        assert err < 1e-10, (key, err)
    _, _, states = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                  d["h0"], cu_seqlens=cu, chunk=C, want_chunk_states=True)
    np.testing.assert_allclose(got["states"], states, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got["dstates"], ref["chunk_dstates"], rtol=1e-10, atol=1e-12)


def test_chunked_equals_token_serial_with_gate_bias():
    rng = np.random.default_rng(3)
    cu = [0, 1, 63, 128, 193]
    H, K, V = 2, 8, 6
    d = _inputs(rng, cu[-1], H, K, V, len(cu) - 1)
    b = rng.standard_normal((H, K))
    ref = oracle.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                          d["dO"], d["dhT"], cu_seqlens=cu, chunk=16, dt_bias=b)
    got = chunked.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["h0"],
                           d["dO"], d["dhT"], cu_seqlens=cu, chunk=16, dt_bias=b)
    for key in KEYS + ("ddt_bias",):
        err = np.linalg.norm(got[key] - ref[key]) / np.linalg.norm(ref[key])
        assert err < 1e-10, (key, err)
