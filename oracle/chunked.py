"""Chunked (WY / UT-transform) restatement of the KDA forward and backward in
fp64 numpy -- TEST INFRASTRUCTURE ONLY.

This is a second CPU formulation, written independently of the token-serial
C oracle, of the chunk algebra the GPU kernels follow.  The tests require it
to equal the token-serial oracle to ~1e-10 for several chunk sizes; that pins
the algebra (the WY inverse, the intra-chunk masks, the reverse state-gradient
scan and the per-chunk gradient terms) without sharing any code with the CUDA
path.  fp64 has the range to form k * exp(-gc) directly, so no sub-block
re-referencing is needed here.

Per chunk (rows i, j; gc the within-chunk running sum of gk, gT its last row;
the names follow the kernel-B guide, "bwd-kernelB-beginner-guide-full",
Part 2: kd / ki / kr are the decayed, inverse-decayed and end-decayed keys):

  qd = q^ e^gc,  kd = k^ e^gc,  ki = k^ e^-gc,  kr = k^ e^(gT - gc)
  Akk = strict_lower(diag(beta) kd ki^T),  INV = (I + Akk)^-1
  Mqk = lower_incl(qd ki^T)
  U   = INV (beta * (v - kd S_n))                     (v_new)
  O   = s (qd S_n + Mqk U)
  S_{n+1} = diag(e^gT) S_n + kr^T U

Backward of one chunk, given dO and dS_{n+1} (Kernel A / Kernel B split of
the bwd-ncu-and-optimization-playbook, A/B table):

  dU     = s Mqk^T dO + kr dS_{n+1}                     (B1: dU)
  dvcorr = INV^T dU                                      (B1: dvcorr)
  dS_n   = diag(e^gT) dS_{n+1} + s qd^T dO - (beta kd)^T dvcorr
  dv     = beta dvcorr                                   (B1: dv)
  dbeta  = rowsum(dvcorr (v - kd S_n)) + rowsum(dAkk * kd ki^T)   (B2: dbeta)
  dMqk   = lower_incl(s dO U^T);  dAkk = -strict_lower(dvcorr U^T)
  dqd    = s dO S_n^T + dMqk ki                          (B2: dqd)
  dkd    = -diag(beta) dvcorr S_n^T + diag(beta) dAkk ki (B2: dkd)
  dki    = dMqk^T qd + (diag(beta) dAkk)^T kd
  dkr    = U dS_{n+1}^T                                  (B1: dkr)
  dgc    = dqd qd + dkd kd - dki ki - dkr kr            (B3: gate-gradient)
  dgT    = e^gT rowdot(dS_{n+1}, S_n) + colsum(dkr kr)  (B0: dgT-dot)
  dgk    = reverse_cumsum(dgc) + dgT                     (B3/K1 reverse cumsum)
  dq^    = dqd e^gc;  dk^ = dkd e^gc + dki e^-gc + dkr e^(gT - gc)
"""
from __future__ import annotations

import numpy as np


def _softplus(x):
    return np.logaddexp(0.0, x)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _unit_chunks(L, C):
    return [(a, min(a + C, L)) for a in range(0, L, C)]


def backward(q, k, v, g, beta, A_log, h0, dO, dhT, *, cu_seqlens, scale=None,
             eps=1e-6, chunk=64, dt_bias=None):
    """Chunked fp64 backward (and the forward states it needs).

    ``dt_bias`` (optional ``[H, K]``) enters the gate as softplus(g + dt_bias).
    Returns a dict with dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0 and the per-chunk
    intermediates ``states`` (S_n, state at chunk start) and ``dstates``
    (dS_{n+1}, adjoint of the state at chunk end), both ``[NTc, H, K, V]``.
    """
    q, k, v, g, beta, dO = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, dO))
    A_log = np.asarray(A_log, dtype=np.float64)
    Ttot, H, K = q.shape
    V = v.shape[2]
    s = K ** -0.5 if scale is None else scale
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    C = chunk
    nck = [(int(cu[i + 1] - cu[i]) + C - 1) // C for i in range(N)]
    base = np.concatenate([[0], np.cumsum(nck)]).astype(np.int64)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dg=np.zeros_like(g), dbeta=np.zeros_like(beta),
               dA_log=np.zeros(H), ddt_bias=np.zeros((H, K)), dh0=np.zeros((N, H, K, V)),
               states=np.zeros((int(base[-1]), H, K, V)),
               dstates=np.zeros((int(base[-1]), H, K, V)))
    for sq in range(N):
        t0, L = int(cu[sq]), int(cu[sq + 1] - cu[sq])
        for h in range(H):
            A = np.exp(A_log[h])
            rows = slice(t0, t0 + L)
            qh, kh = q[rows, h], k[rows, h]
            gh = g[rows, h] + (0.0 if dt_bias is None else np.asarray(dt_bias, np.float64)[h])
            nq = np.sqrt((qh ** 2).sum(-1, keepdims=True) + eps)
            nk = np.sqrt((kh ** 2).sum(-1, keepdims=True) + eps)
            qn, kn = qh / nq, kh / nk
            gk = -A * _softplus(gh)
            vh, bh, dOh = v[rows, h], beta[rows, h], dO[rows, h]
            S = np.zeros((K, V)) if h0 is None else np.array(h0[sq, h], dtype=np.float64)
            per = []
            # forward over chunks: states and the per-chunk operands
            for ci, (a, b) in enumerate(_unit_chunks(L, C)):
                n = b - a
                gc = np.cumsum(gk[a:b], 0)
                gT = gc[-1]
                qd = qn[a:b] * np.exp(gc)
                kd = kn[a:b] * np.exp(gc)
                ki = kn[a:b] * np.exp(-gc)
                kr = kn[a:b] * np.exp(gT - gc)
                bb = bh[a:b]
                Gkk = kd @ ki.T
                Akk = np.tril(bb[:, None] * Gkk, -1)
                INV = np.linalg.inv(np.eye(n) + Akk)
                Mqk = np.tril(qd @ ki.T)
                X = vh[a:b] - kd @ S
                U = INV @ (bb[:, None] * X)
                out["states"][base[sq] + ci, h] = S
                per.append(dict(a=a, b=b, gc=gc, gT=gT, qd=qd, kd=kd, ki=ki, kr=kr,
                                bb=bb, Gkk=Gkk, INV=INV, Mqk=Mqk, X=X, U=U, S=S))
                S = np.exp(gT)[:, None] * S + kr.T @ U
            # reverse over chunks
            dS = np.zeros((K, V)) if dhT is None else np.array(dhT[sq, h], dtype=np.float64)
            dqn = np.zeros_like(qn)
            dkn = np.zeros_like(kn)
            dgk = np.zeros_like(gk)
            for ci in range(len(per) - 1, -1, -1):
                c = per[ci]
                a, b = c["a"], c["b"]
                out["dstates"][base[sq] + ci, h] = dS
                dOc = dOh[a:b]
                Sn = c["S"]
                dU = s * c["Mqk"].T @ dOc + c["kr"] @ dS
                dvcorr = c["INV"].T @ dU
                dMqk = np.tril(s * dOc @ c["U"].T)
                dAkk = -np.tril(dvcorr @ c["U"].T, -1)
                dA = c["bb"][:, None] * dAkk
                dqd = s * dOc @ Sn.T + dMqk @ c["ki"]
                dkd = -c["bb"][:, None] * (dvcorr @ Sn.T) + dA @ c["ki"]
                dki = dMqk.T @ c["qd"] + dA.T @ c["kd"]
                dkr = c["U"] @ dS.T
                out["dv"][t0 + a:t0 + b, h] = c["bb"][:, None] * dvcorr
                out["dbeta"][t0 + a:t0 + b, h] = ((dvcorr * c["X"]).sum(-1)
                                                  + (dAkk * c["Gkk"]).sum(-1))
                dgc = dqd * c["qd"] + dkd * c["kd"] - dki * c["ki"] - dkr * c["kr"]
                dgT = np.exp(c["gT"]) * (dS * Sn).sum(-1) + (dkr * c["kr"]).sum(0)
                dgk[a:b] = np.cumsum(dgc[::-1], 0)[::-1] + dgT[None, :]
                dqn[a:b] = dqd * np.exp(c["gc"])
                dkn[a:b] = (dkd * np.exp(c["gc"]) + dki * np.exp(-c["gc"])
                            + dkr * np.exp(c["gT"] - c["gc"]))
                dS = (np.exp(c["gT"])[:, None] * dS + s * c["qd"].T @ dOc
                      - (c["bb"][:, None] * c["kd"]).T @ dvcorr)
            out["dh0"][sq, h] = dS
            out["dq"][rows, h] = (dqn - qn * (qn * dqn).sum(-1, keepdims=True)) / nq
            out["dk"][rows, h] = (dkn - kn * (kn * dkn).sum(-1, keepdims=True)) / nk
            out["dg"][rows, h] = dgk * (-A) * _sigmoid(gh)
            out["ddt_bias"][h] += out["dg"][rows, h].sum(0)
            out["dA_log"][h] += np.sum(dgk * gk)
    return out
