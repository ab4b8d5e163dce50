"""Chunkwise (WY / UT-transform) form of the KDA gated delta rule, fp64 numpy.

Test helper. It restates the recurrence in the chunked form the CUDA kernels
use, so that two independent formulations (this one and the token-by-token
oracle) can pin each other, and it documents the chunk algebra and its
hand-derived adjoints.

Within a chunk of L <= C tokens starting from state S0 (V x K), with
G = cumsum(g) (per key channel), Gam = exp(G):
  A_ij   = beta_i sum_c k^_ic k^_jc e^{G_ic - G_jc}     (j < i)
  Aqk_ij = sum_c q^_ic k^_jc e^{G_ic - G_jc}            (j <= i)
  T = (I + A)^{-1} diag(beta),  W = T (K^ * Gam),  U = T V
  Ut = U - W S0^T
  O  = scale [ (Q^ * Gam) S0^T + Aqk Ut ]
  S_L = S0 diag(e^{G_L}) + Ut^T (K^ * e^{G_L - G})
(the kda-neuron-kernels log calls this the exact "16-sub-chunk + WY" form;
its chunk size here is a parameter).
"""
from __future__ import annotations

import numpy as np

SCALE = 1.0 / np.sqrt(128.0)
LB = -5.0
EPS = 1e-6


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _prep(inp, mode):
    q, k, v = _f64(inp["q"]), _f64(inp["k"]), _f64(inp["v"])
    gx, bx = _f64(inp["g_raw"]), _f64(inp["beta_raw"])
    lb = float(inp.get("lower_bound", LB))
    if mode == "raw":
        nq = np.sqrt((q * q).sum(-1, keepdims=True) + EPS)
        nk = np.sqrt((k * k).sum(-1, keepdims=True) + EPS)
        A_log, dt = _f64(inp["A_log"]), _f64(inp["dt_bias"])
        a = np.exp(A_log)[None, :, None]
        s = _sigmoid(a * (gx + dt[None]))
        g = lb * s
        beta = _sigmoid(bx)
        return dict(qh=q / nq, kh=k / nk, v=v, g=g, beta=beta, nq=nq, nk=nk, s=s, a=a,
                    gx=gx, dt=dt, lb=lb)
    return dict(qh=q, kh=k, v=v, g=gx, beta=bx)


def _pair_decay(G):
    """D[i, j, c] = exp(G_ic - G_jc) for j <= i, 0 above the diagonal."""
    L = G.shape[0]
    diff = G[:, None, :] - G[None, :, :]
    mask = np.tril(np.ones((L, L), dtype=bool))
    diff = np.where(mask[:, :, None], diff, -np.inf)
    return np.exp(diff)


def _chunk_fwd(qh, kh, v, g, beta, S0, scale):
    L = qh.shape[0]
    G = np.cumsum(g, axis=0)
    Gam = np.exp(G)
    GL = G[L - 1]
    D = _pair_decay(G)
    Bm = np.einsum("ic,jc,ijc->ij", kh, kh, D) * np.tril(np.ones((L, L)), -1)
    Am = beta[:, None] * Bm
    Aqk = np.einsum("ic,jc,ijc->ij", qh, kh, D)
    X = np.linalg.inv(np.eye(L) + Am)
    Tm = X * beta[None, :]
    Kt = kh * Gam
    W = Tm @ Kt
    U = Tm @ v
    Ut = U - W @ S0.T
    Qb = qh * Gam
    O = scale * (Qb @ S0.T + Aqk @ Ut)
    Kb = kh * np.exp(GL[None, :] - G)
    S1 = S0 * np.exp(GL)[None, :] + Ut.T @ Kb
    ctx = dict(G=G, Gam=Gam, GL=GL, D=D, Bm=Bm, Aqk=Aqk, X=X, Tm=Tm, Kt=Kt, W=W, Ut=Ut,
               Qb=Qb, Kb=Kb, S0=S0)
    return O, S1, ctx


def _chunk_bwd(qh, kh, v, beta, dO, dS1, ctx, scale):
    """Adjoints of one chunk. Returns dqh, dkh, dv, dg, dbeta, dS0."""
    L = qh.shape[0]
    G, Gam, GL, D = ctx["G"], ctx["Gam"], ctx["GL"], ctx["D"]
    Bm, Aqk, X, Tm = ctx["Bm"], ctx["Aqk"], ctx["X"], ctx["Tm"]
    Kt, W, Ut, Qb, Kb, S0 = ctx["Kt"], ctx["W"], ctx["Ut"], ctx["Qb"], ctx["Kb"], ctx["S0"]
    tri_incl = np.tril(np.ones((L, L)))
    tri_strict = np.tril(np.ones((L, L)), -1)

    dUt = scale * Aqk.T @ dO + Kb @ dS1.T
    dQb = scale * dO @ S0
    dAqk = scale * (dO @ Ut.T) * tri_incl
    dKb = Ut @ dS1
    dS0 = dS1 * np.exp(GL)[None, :] + scale * dO.T @ Qb - dUt.T @ W
    dGL = (dS1 * S0).sum(0) * np.exp(GL)
    dW = -dUt @ S0
    dT = dW @ Kt.T + dUt @ v.T
    dKt = Tm.T @ dW
    dv = Tm.T @ dUt
    dbeta = (dT * X).sum(0)
    dA = -(X.T @ (dT @ Tm.T)) * tri_strict
    dbeta = dbeta + (dA * Bm).sum(1)
    dB = beta[:, None] * dA

    dqh = dQb * Gam
    dkh = dKt * Gam + dKb * np.exp(GL[None, :] - G)
    dG = dQb * Qb + dKt * Kt - dKb * Kb
    dGL = dGL + (dKb * Kb).sum(0)
    # pairwise terms: P[i,j,c] = x_ic k_jc D_ijc, with x = k^ (for B) or q^ (for Aqk)
    for dM, xh in ((dB, kh), (dAqk, qh)):
        R = dM[:, :, None] * D                      # [i, j, c]
        dxi = np.einsum("ijc,jc->ic", R, kh)        # sum_j dM_ij k_j D_ij
        dkj = np.einsum("ijc,ic->jc", R, xh)        # sum_i dM_ij x_i D_ij
        if xh is kh:
            dkh = dkh + dxi + dkj
        else:
            dqh = dqh + dxi
            dkh = dkh + dkj
        dG = dG + xh * dxi - kh * dkj
    dG[L - 1] += dGL
    dg = np.flip(np.cumsum(np.flip(dG, 0), 0), 0)
    return dqh, dkh, dv, dg, dbeta, dS0


def _units(inp):
    cu = np.asarray(inp["cu_seqlens"], dtype=np.int64)
    return [(int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]


def forward(inp, C: int = 64, mode: str = "raw"):
    p = _prep(inp, mode)
    scale = float(inp.get("scale", SCALE))
    T, H, K = p["qh"].shape
    V = p["v"].shape[2]
    spans = _units(inp)
    h0 = _f64(inp.get("h0"))
    o = np.zeros((T, H, V))
    hT = np.zeros((len(spans), H, V, K))
    for n, (b, e) in enumerate(spans):
        for h in range(H):
            S = h0[n, h].copy() if h0 is not None else np.zeros((V, K))
            for c0 in range(b, e, C):
                c1 = min(c0 + C, e)
                O, S, _ = _chunk_fwd(p["qh"][c0:c1, h], p["kh"][c0:c1, h], p["v"][c0:c1, h],
                                     p["g"][c0:c1, h], p["beta"][c0:c1, h], S, scale)
                o[c0:c1, h] = O
            hT[n, h] = S
    return dict(o=o, hT=hT)


def backward(inp, C: int = 64, mode: str = "raw"):
    p = _prep(inp, mode)
    scale = float(inp.get("scale", SCALE))
    T, H, K = p["qh"].shape
    V = p["v"].shape[2]
    spans = _units(inp)
    h0, dhT, dO = _f64(inp.get("h0")), _f64(inp.get("dhT")), _f64(inp["do"])
    dqh = np.zeros((T, H, K)); dkh = np.zeros((T, H, K)); dv = np.zeros((T, H, V))
    dg = np.zeros((T, H, K)); dbeta = np.zeros((T, H)); dh0 = np.zeros((len(spans), H, V, K))
    for n, (b, e) in enumerate(spans):
        for h in range(H):
            S = h0[n, h].copy() if h0 is not None else np.zeros((V, K))
            ctxs = []
            for c0 in range(b, e, C):
                c1 = min(c0 + C, e)
                _, S, ctx = _chunk_fwd(p["qh"][c0:c1, h], p["kh"][c0:c1, h], p["v"][c0:c1, h],
                                       p["g"][c0:c1, h], p["beta"][c0:c1, h], S, scale)
                ctxs.append((c0, c1, ctx))
            dS = dhT[n, h].copy() if dhT is not None else np.zeros((V, K))
            for c0, c1, ctx in reversed(ctxs):
                r = _chunk_bwd(p["qh"][c0:c1, h], p["kh"][c0:c1, h], p["v"][c0:c1, h],
                               p["beta"][c0:c1, h], dO[c0:c1, h], dS, ctx, scale)
                dqh[c0:c1, h], dkh[c0:c1, h], dv[c0:c1, h] = r[0], r[1], r[2]
                dg[c0:c1, h], dbeta[c0:c1, h], dS = r[3], r[4], r[5]
            dh0[n, h] = dS
    out = dict(dv=dv, dh0=dh0)
    if mode != "raw":
        out.update(dq=dqh, dk=dkh, dg_raw=dg, dbeta_raw=dbeta)
        return out
    # chains: L2 norm, gate, beta sigmoid
    qh, kh, nq, nk = p["qh"], p["kh"], p["nq"], p["nk"]
    out["dq"] = (dqh - qh * (qh * dqh).sum(-1, keepdims=True)) / nq
    out["dk"] = (dkh - kh * (kh * dkh).sum(-1, keepdims=True)) / nk
    du = dg * p["lb"] * p["s"] * (1.0 - p["s"])
    out["dg_raw"] = du * p["a"]
    out["ddt_bias"] = out["dg_raw"].sum(0)
    out["dA_log"] = (out["dg_raw"] * (p["gx"] + p["dt"][None])).sum((0, 2))
    out["dbeta_raw"] = dbeta * p["beta"] * (1.0 - p["beta"])
    return out
