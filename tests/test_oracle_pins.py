"""Pins of the fp64 CPU oracle against facts that do not come from the oracle.

* central finite differences of the oracle's own forward (pins the reverse
  mode, every input, including the erase term, h0 and varlen boundaries);
* closed forms: beta = 0 (pure per-channel decay of h0), the erase-off
  ablation with beta = 1 (gated linear attention) and, with zero decay,
  causal linear attention in matrix form with its textbook gradients;
* the basis-key overwrite invariant of the delta rule;
* linearity of the VJP in the cotangents, varlen == separate calls,
  head permutation equivariance.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
sign, a transposed operand, an off-by-one in the token index) fails it.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def _rand_inputs(rng, Ttot, H, K, V, N=1, h0=True, dhT=True):
    d = dict(
        q=rng.standard_normal((Ttot, H, K)),
        k=rng.standard_normal((Ttot, H, K)),
        v=rng.standard_normal((Ttot, H, V)),
        g=rng.standard_normal((Ttot, H, K)),
        beta=1.0 / (1.0 + np.exp(-rng.standard_normal((Ttot, H)))),
        A_log=rng.uniform(0.0, 1.5, size=(H,)),
        h0=0.5 * rng.standard_normal((N, H, K, V)) if h0 else None,
        dO=rng.standard_normal((Ttot, H, V)),
        dhT=rng.standard_normal((N, H, K, V)) if dhT else None,
    )
    return d


def _loss(inp, cu, **kw):
    o, hT, _ = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"],
                              inp["beta"], inp["A_log"], inp["h0"],
                              cu_seqlens=cu, dt_bias=inp.get("dt_bias"), **kw)
    L = float(np.sum(o * inp["dO"]))
    if inp["dhT"] is not None:
        L += float(np.sum(hT * inp["dhT"]))
    return L


def _grads(inp, cu, **kw):
    return oracle.backward(inp["q"], inp["k"], inp["v"], inp["g"],
                           inp["beta"], inp["A_log"], inp["h0"], inp["dO"],
                           inp["dhT"], cu_seqlens=cu, dt_bias=inp.get("dt_bias"), **kw)


GRAD_OF = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", A_log="dA_log",
               h0="dh0", dt_bias="ddt_bias")


def _fd_check(inp, cu, max_elems=48, step=1e-6, tol=1e-6, rng=RNG, **kw):
    an = _grads(inp, cu, **kw)
    for name, gname in GRAD_OF.items():
        if inp.get(name) is None:
            continue
        x = inp[name]
        flat = x.reshape(-1)
        idx = np.arange(flat.size)
        if flat.size > max_elems:
            idx = rng.choice(flat.size, size=max_elems, replace=False)
        fd = np.empty(len(idx))
        for n, i in enumerate(idx):
            old = flat[i]
            flat[i] = old + step
            lp = _loss(inp, cu, **kw)
            flat[i] = old - step
            lm = _loss(inp, cu, **kw)
            flat[i] = old
            fd[n] = (lp - lm) / (2 * step)
        a = an[gname].reshape(-1)[idx]
        err = np.linalg.norm(fd - a) / max(np.linalg.norm(a), 1e-30)
        assert err <= tol, f"{name}: FD rel err {err:.3e} (|grad|={np.linalg.norm(a):.3e})"


@pytest.mark.parametrize("T,K,chunk", [(1, 2, 64), (5, 4, 64), (17, 8, 4),
                                       (70, 4, 64), (70, 8, 16)])
def test_fd_full_vjp(T, K, chunk):
    rng = np.random.default_rng(T * 100 + K)
    inp = _rand_inputs(rng, T, 2, K, K)
    _fd_check(inp, [0, T], chunk=chunk, rng=rng)


def test_fd_rectangular_heads():
    rng = np.random.default_rng(7)
    inp = _rand_inputs(rng, 9, 2, 4, 6)  # K != V catches transposed operands
    _fd_check(inp, [0, 9], chunk=4, rng=rng)


def test_fd_varlen_boundaries():
    rng = np.random.default_rng(11)
    cu = [0, 5, 17, 18, 26]
    inp = _rand_inputs(rng, 26, 2, 4, 4, N=4)
    _fd_check(inp, cu, chunk=4, rng=rng)


def test_fd_erase_off_and_raw_gate():
    rng = np.random.default_rng(5)
    inp = _rand_inputs(rng, 12, 2, 4, 4)
    inp["g"] = -np.abs(inp["g"])
    _fd_check(inp, [0, 12], chunk=4, gate_mode=1, erase=0, rng=rng)


def test_fd_gate_bias():
    # the gate's per-channel bias: gk = -exp(A_log) softplus(g + dt_bias)
    rng = np.random.default_rng(17)
    cu = [0, 7, 19, 20]
    inp = _rand_inputs(rng, 20, 2, 4, 5, N=3)
    inp["dt_bias"] = rng.standard_normal((2, 4))
    _fd_check(inp, cu, chunk=4, rng=rng)


def test_gate_bias_is_a_shift_of_g():
    # the bias only shifts g inside softplus: (g, b) and (g + b, 0) are the
    # same model with the same gradients (ddt_bias included, it is the sum of
    # dg); and no bias at all equals a zero bias
    rng = np.random.default_rng(19)
    cu = [0, 9, 30]
    inp = _rand_inputs(rng, 30, 2, 4, 4, N=2)
    b = rng.standard_normal((2, 4))
    ref = _grads(dict(inp, dt_bias=b), cu, chunk=8)
    shifted = dict(inp, g=inp["g"] + b[None], dt_bias=np.zeros((2, 4)))
    got = _grads(shifted, cu, chunk=8)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "dh0", "ddt_bias"):
        np.testing.assert_allclose(got[key], ref[key], rtol=1e-12, atol=1e-12)
    plain = _grads(inp, cu, chunk=8)
    zero = _grads(dict(inp, dt_bias=np.zeros((2, 4))), cu, chunk=8)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "dh0", "ddt_bias"):
        np.testing.assert_array_equal(plain[key], zero[key])


def test_beta_zero_closed_form():
    """beta = 0: S_t = Diag(exp(G_t)) h0 with G_t the running sum of gk."""
    rng = np.random.default_rng(3)
    T, H, K, V = 23, 2, 5, 3
    inp = _rand_inputs(rng, T, H, K, V)
    inp["beta"][:] = 0.0
    scale = 0.37
    o, hT, _ = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"],
                              inp["beta"], inp["A_log"], inp["h0"],
                              cu_seqlens=[0, T], scale=scale)
    gr = _grads(inp, [0, T], scale=scale)
    eps = 1e-6
    for h in range(H):
        A = np.exp(inp["A_log"][h])
        gk = -A * np.logaddexp(0.0, inp["g"][:, h, :])          # [T, K]
        G = np.cumsum(gk, axis=0)                                 # [T, K]
        qn = inp["q"][:, h] / np.sqrt((inp["q"][:, h] ** 2).sum(-1, keepdims=True) + eps)
        kn = inp["k"][:, h] / np.sqrt((inp["k"][:, h] ** 2).sum(-1, keepdims=True) + eps)
        h0 = inp["h0"][0, h]
        S = np.exp(G)[:, :, None] * h0[None]                      # S_t, [T, K, V]
        np.testing.assert_allclose(o[:, h], scale * np.einsum("tk,tkv->tv", qn, S), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(hT[0, h], S[-1], rtol=1e-12, atol=1e-14)
        assert np.all(gr["dv"][:, h] == 0.0) and np.all(gr["dk"][:, h] == 0.0)
        # adjoint of S_t: everything read at tau >= t, decayed back to t
        dO = inp["dO"][:, h]
        adj = np.zeros((T, K, V))
        for t in range(T):
            acc = np.exp(G[-1] - G[t])[:, None] * inp["dhT"][0, h]
            for tau in range(t, T):
                acc = acc + scale * np.exp(G[tau] - G[t])[:, None] * np.outer(qn[tau], dO[tau])
            adj[t] = acc
        dh0 = np.exp(G[0])[:, None] * adj[0]
        np.testing.assert_allclose(gr["dh0"][0, h], dh0, rtol=1e-11, atol=1e-13)
        Sprev = np.concatenate([h0[None], S[:-1]], 0)
        Sp = np.exp(gk)[:, :, None] * Sprev                       # S'_t
        delta = inp["v"][:, h] - np.einsum("tkv,tk->tv", Sp, kn)
        dbeta = np.einsum("tk,tkv,tv->t", kn, adj, delta)
        np.testing.assert_allclose(gr["dbeta"][:, h], dbeta, rtol=1e-11, atol=1e-13)
        dqn = scale * np.einsum("tkv,tv->tk", S, dO)
        nq = np.sqrt((inp["q"][:, h] ** 2).sum(-1, keepdims=True) + eps)
        dq = (dqn - qn * (qn * dqn).sum(-1, keepdims=True)) / nq
        np.testing.assert_allclose(gr["dq"][:, h], dq, rtol=1e-11, atol=1e-13)


def test_causal_linear_attention_closed_form():
    """erase off, beta = 1, zero decay, no norm: o = s tril(Q K^T) V + s Q h0."""
    rng = np.random.default_rng(9)
    T, H, K, V = 19, 2, 6, 4
    inp = _rand_inputs(rng, T, H, K, V)
    inp["beta"][:] = 1.0
    inp["g"][:] = 0.0
    s = 0.5
    kw = dict(scale=s, gate_mode=1, erase=0, normalize=0)
    o, hT, _ = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"],
                              inp["beta"], inp["A_log"], inp["h0"],
                              cu_seqlens=[0, T], **kw)
    gr = _grads(inp, [0, T], **kw)
    M = np.tril(np.ones((T, T)))
    for h in range(H):
        Q, Kk, Vv = inp["q"][:, h], inp["k"][:, h], inp["v"][:, h]
        h0, dhT, dO = inp["h0"][0, h], inp["dhT"][0, h], inp["dO"][:, h]
        P = M * (Q @ Kk.T)
        np.testing.assert_allclose(o[:, h], s * (P @ Vv + Q @ h0), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(hT[0, h], h0 + Kk.T @ Vv, rtol=1e-12, atol=1e-12)
        dP = M * (dO @ Vv.T)
        np.testing.assert_allclose(gr["dv"][:, h], s * P.T @ dO + Kk @ dhT, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(gr["dq"][:, h], s * (dP @ Kk + dO @ h0.T), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(gr["dk"][:, h], s * dP.T @ Q + Vv @ dhT.T, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(gr["dh0"][0, h], s * Q.T @ dO + dhT, rtol=1e-11, atol=1e-12)
        dbeta = np.einsum("tk,tkv,tv->t", Kk, _adj_nodecay(Q, dO, dhT, s), Vv)
        np.testing.assert_allclose(gr["dbeta"][:, h], dbeta, rtol=1e-11, atol=1e-12)


def _adj_nodecay(Q, dO, dhT, s):
    T = Q.shape[0]
    adj = np.zeros((T,) + dhT.shape)
    acc = dhT.copy()
    for t in range(T - 1, -1, -1):
        acc = acc + s * np.outer(Q[t], dO[t])
        adj[t] = acc
    return adj


def test_gated_linear_attention_forward():
    """erase off, beta = 1: o_t = s sum_{j<=t} (q_t * exp(G_t - G_j)) . k_j v_j + s (q_t * exp(G_t))^T h0."""
    rng = np.random.default_rng(21)
    T, H, K, V = 14, 2, 5, 3
    inp = _rand_inputs(rng, T, H, K, V)
    inp["beta"][:] = 1.0
    s = 0.3
    o, _, _ = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"],
                             inp["beta"], inp["A_log"], inp["h0"],
                             cu_seqlens=[0, T], scale=s, erase=0, normalize=0)
    for h in range(H):
        gk = -np.exp(inp["A_log"][h]) * np.logaddexp(0.0, inp["g"][:, h])
        G = np.cumsum(gk, 0)
        Q, Kk, Vv = inp["q"][:, h], inp["k"][:, h], inp["v"][:, h]
        for t in range(T):
            ref = s * (Q[t] * np.exp(G[t])) @ inp["h0"][0, h]
            for j in range(t + 1):
                ref = ref + s * np.sum(Q[t] * np.exp(G[t] - G[j]) * Kk[j]) * Vv[j]
            np.testing.assert_allclose(o[t, h], ref, rtol=1e-12, atol=1e-13)


def test_basis_key_overwrite():
    """k_t one-hot, beta = 1, no decay, h0 = 0: row i of S is the last v
    written under key i, so o_t = s sum_i q_t[i] v_last(i, <= t)."""
    rng = np.random.default_rng(4)
    T, K, V = 40, 6, 5
    keys = rng.integers(0, K, size=T)
    q = rng.standard_normal((T, 1, K))
    k = np.zeros((T, 1, K))
    k[np.arange(T), 0, keys] = 1.0
    v = rng.standard_normal((T, 1, V))
    s = 0.7
    o, hT, _ = oracle.forward(q, k, v, np.zeros((T, 1, K)), np.ones((T, 1)),
                              np.zeros(1), None, cu_seqlens=[0, T], scale=s,
                              gate_mode=1, normalize=0)
    last = np.zeros((K, V))
    for t in range(T):
        last[keys[t]] = v[t, 0]
        np.testing.assert_allclose(o[t, 0], s * q[t, 0] @ last, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hT[0, 0], last, rtol=1e-13, atol=1e-14)


def test_linearity_in_cotangents():
    rng = np.random.default_rng(8)
    T, H, K = 21, 2, 4
    inp = _rand_inputs(rng, T, H, K, K)
    dO2 = rng.standard_normal(inp["dO"].shape)
    dh2 = rng.standard_normal(inp["dhT"].shape)
    a, b = 0.7, -1.3
    g1 = _grads(inp, [0, T], chunk=8)
    inp2 = dict(inp, dO=dO2, dhT=dh2)
    g2 = _grads(inp2, [0, T], chunk=8)
    inp3 = dict(inp, dO=a * inp["dO"] + b * dO2, dhT=a * inp["dhT"] + b * dh2)
    g3 = _grads(inp3, [0, T], chunk=8)
    for key in GRAD_OF.values():
        np.testing.assert_allclose(g3[key], a * g1[key] + b * g2[key], rtol=1e-10, atol=1e-12)


def test_varlen_equals_separate_calls():
    rng = np.random.default_rng(12)
    cu = [0, 7, 7, 30, 31]
    H, K = 2, 4
    inp = _rand_inputs(rng, 31, H, K, K, N=4)
    packed = _grads(inp, cu, chunk=8)
    o_p, hT_p, _ = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                  inp["A_log"], inp["h0"], cu_seqlens=cu, chunk=8)
    dA = np.zeros(H)
    for s in range(4):
        a, b = cu[s], cu[s + 1]
        sub = {n: (x[a:b] if n in ("q", "k", "v", "g", "beta", "dO") else x)
               for n, x in inp.items()}
        sub["h0"] = inp["h0"][s:s + 1]
        sub["dhT"] = inp["dhT"][s:s + 1]
        gs = _grads(sub, [0, b - a], chunk=8)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            assert np.array_equal(gs[key], packed[key][a:b]), key
        assert np.array_equal(gs["dh0"][0], packed["dh0"][s])
        o_s, hT_s, _ = oracle.forward(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                      sub["A_log"], sub["h0"], cu_seqlens=[0, b - a], chunk=8)
        assert np.array_equal(o_s, o_p[a:b]) and np.array_equal(hT_s[0], hT_p[s])
        dA += gs["dA_log"]
    np.testing.assert_allclose(packed["dA_log"], dA, rtol=1e-13)


def test_head_permutation():
    rng = np.random.default_rng(13)
    T, H, K = 10, 3, 4
    inp = _rand_inputs(rng, T, H, K, K)
    perm = np.array([2, 0, 1])
    g0 = _grads(inp, [0, T])
    pinp = dict(inp)
    for n in ("q", "k", "v", "g", "beta", "dO"):
        pinp[n] = inp[n][:, perm]
    pinp["A_log"] = inp["A_log"][perm]
    pinp["h0"] = inp["h0"][:, perm]
    pinp["dhT"] = inp["dhT"][:, perm]
    g1 = _grads(pinp, [0, T])
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        assert np.array_equal(g1[key], g0[key][:, perm])
    assert np.array_equal(g1["dA_log"], g0["dA_log"][perm])
    assert np.array_equal(g1["dh0"], g0["dh0"][:, perm])


def test_chunk_state_outputs_match_final_state():
    rng = np.random.default_rng(14)
    T, H, K = 20, 2, 4
    inp = _rand_inputs(rng, T, H, K, K)
    o, hT, cs = oracle.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                               inp["A_log"], inp["h0"], cu_seqlens=[0, T], chunk=8,
                               want_chunk_states=True)
    assert cs.shape == (3, H, K, K)
    np.testing.assert_array_equal(cs[0], inp["h0"][0])
    _, hT8, _ = oracle.forward(inp["q"][:8], inp["k"][:8], inp["v"][:8], inp["g"][:8],
                               inp["beta"][:8], inp["A_log"], inp["h0"], cu_seqlens=[0, 8])
    np.testing.assert_array_equal(cs[1], hT8[0])
    gr = _grads(inp, [0, T], chunk=8, want_chunk_dstates=True)
    np.testing.assert_array_equal(gr["chunk_dstates"][2], inp["dhT"][0])
