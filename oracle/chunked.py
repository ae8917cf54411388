"""Chunk-parallel form of KDA in fp64 numpy (test infrastructure only).

This is the same computation as the token recurrence in ``kda_oracle.c``,
regrouped into chunks of C tokens the way the chunked kernels do it. It
follows, in the notation used across this package,

* the chunked forward that the FlashKDA backward page (K2) recomputes
  ("Step 1: Recompute U": vcorr = beta (v - K~ S_in), U = INV vcorr with
  INV = (I + L)^-1, L = tril(K~ K^T, -1) * beta; S_new = S exp(gT) + K^T U),
* the data flow of FLA's ``chunk_kda_bwd`` (the ``chunk_bwd.py`` page):
  recompute w, u; state pass storing h = S_in per chunk; dAqk = scale
  tril(dO v_new^T) and dv = Aqk^T dO (kernel ``dAv``); the reverse dh pass;
  the fused w/y kernel (dq = dO h^T e^G scale, dk = v_new dh^T e^(G_C - G),
  dw = -dv h^T, dA = -A^T (dA (.) beta) A^T on the strict lower triangle, dg =
  q dq - k dk + [last row] dgk + kg dkgb beta); the triangle backward; and
  the final in-chunk reverse cumsum of dg.

Within one chunk of c valid rows (Gamma_r = sum_{s<=r} g_s, natural log)::

    K~ = k e^Gamma,   Q~ = q e^Gamma,   K^ = k e^(Gamma_C - Gamma)
    Akk[r,j] = beta_r sum_d k_rd k_jd e^(Gamma_rd - Gamma_jd)        (j < r)
    Aqk[r,j] = scale  sum_d q_rd k_jd e^(Gamma_rd - Gamma_jd)        (j <= r)
    INV = (I + Akk)^-1,  u = INV diag(beta) V,  w = INV diag(beta) K~
    delta = u - w S_in
    O = scale Q~ S_in + Aqk delta
    S_out = Diag(e^Gamma_C) S_in + K^^T delta

The decayed triangles are formed from the exponent differences directly (no
e^Gamma * e^-Gamma factorisation), so the oracle has no overflow limit of its
own. The backward is reverse mode of the same expressions.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular

from . import _f64


def _tri(c, strict):
    return np.tril(np.ones((c, c)), -1 if strict else 0)


def _decay(Gam):
    """D[r, j, d] = exp(Gamma_rd - Gamma_jd) for j <= r, else 0."""
    c = Gam.shape[0]
    le = _tri(c, False).astype(bool)[:, :, None]
    diff = np.where(le, Gam[:, None, :] - Gam[None, :, :], 0.0)
    return np.where(le, np.exp(diff), 0.0)


def chunk_forward(qc, kc, vc, gc, bc, scale, S_in):
    """Per-chunk forward; returns a dict of every intermediate."""
    c = kc.shape[0]
    Gam = np.cumsum(gc, axis=0)
    E = np.exp(Gam)
    GamC = Gam[-1]
    Qt, Kt = qc * E, kc * E
    Kh = kc * np.exp(GamC[None, :] - Gam)
    D = _decay(Gam)
    M = np.einsum("rd,jd,rjd->rj", kc, kc, D) * _tri(c, True)
    Akk = bc[:, None] * M
    Aqk = scale * np.einsum("rd,jd,rjd->rj", qc, kc, D) * _tri(c, False)
    I = np.eye(c)
    INV = solve_triangular(I + Akk, I, lower=True, unit_diagonal=True)
    Xv, Xk = bc[:, None] * vc, bc[:, None] * Kt
    u, w = INV @ Xv, INV @ Xk
    delta = u - w @ S_in
    O = scale * Qt @ S_in + Aqk @ delta
    S_out = np.exp(GamC)[:, None] * S_in + Kh.T @ delta
    return dict(Gamma=Gam, E=E, Qt=Qt, Kt=Kt, Kh=Kh, D=D, M=M, Akk=Akk, Aqk=Aqk, INV=INV, Xv=Xv,
                Xk=Xk, u=u, w=w, delta=delta, O=O, S_in=S_in, S_out=S_out)


def chunk_backward(f, qc, kc, vc, bc, scale, dO, dS_out):
    """Per-chunk backward from the forward intermediates ``f``.

    Returns (dq, dk, dv, dgamma, dbeta, dS_in, extras) for the chunk's rows,
    where dgamma is the gradient w.r.t. the in-chunk cumsum Gamma (the reverse
    cumsum to per-token dg is done by the caller)."""
    c = kc.shape[0]
    Gam, E, Qt, Kt, Kh, D = f["Gamma"], f["E"], f["Qt"], f["Kt"], f["Kh"], f["D"]
    Aqk, INV, w, delta, S_in, M = f["Aqk"], f["INV"], f["w"], f["delta"], f["S_in"], f["M"]
    GamC = Gam[-1]
    EC = np.exp(GamC)
    # o = scale Q~ S_in + Aqk delta ; S_out = e^G_C S_in + K^^T delta
    d_delta = Aqk.T @ dO + Kh @ dS_out
    dS_in = EC[:, None] * dS_out + scale * Qt.T @ dO - w.T @ d_delta
    dQt = scale * dO @ S_in.T
    dAqk = (dO @ delta.T) * _tri(c, False)
    dKh = delta @ dS_out.T
    dGamC = EC * np.sum(S_in * dS_out, axis=1)
    # delta = u - w S_in
    du, dw = d_delta, -d_delta @ S_in.T
    # u = INV Xv, w = INV Xk, INV = (I + Akk)^-1
    dXv, dXk = INV.T @ du, INV.T @ dw
    dINV = du @ f["Xv"].T + dw @ f["Xk"].T
    dAkk = -(INV.T @ dINV @ INV.T) * _tri(c, True)
    dv = bc[:, None] * dXv
    dbeta = np.sum(dXv * vc, axis=1) + np.sum(dXk * Kt, axis=1)
    dKt = bc[:, None] * dXk
    dq = np.zeros_like(qc)
    dk = np.zeros_like(kc)
    dGam = np.zeros_like(Gam)
    # Akk = beta_r * M, M[r,j] = sum_d k_rd k_jd D_rjd (strict lower)
    dbeta += np.sum(dAkk * M, axis=1)
    dM = bc[:, None] * dAkk
    P = kc[:, None, :] * kc[None, :, :] * D
    dk += np.einsum("rj,jd,rjd->rd", dM, kc, D) + np.einsum("rj,rd,rjd->jd", dM, kc, D)
    dGam += np.einsum("rj,rjd->rd", dM, P) - np.einsum("rj,rjd->jd", dM, P)
    # Aqk[r,j] = scale sum_d q_rd k_jd D_rjd (lower incl. diagonal)
    dN = scale * dAqk
    Pq = qc[:, None, :] * kc[None, :, :] * D
    dq += np.einsum("rj,jd,rjd->rd", dN, kc, D)
    dk += np.einsum("rj,rd,rjd->jd", dN, qc, D)
    dGam += np.einsum("rj,rjd->rd", dN, Pq) - np.einsum("rj,rjd->jd", dN, Pq)
    # Q~ = q e^G, K~ = k e^G, K^ = k e^(G_C - G)
    dq += dQt * E
    dGam += dQt * Qt
    dk += dKt * E
    dGam += dKt * Kt
    dk += dKh * np.exp(GamC[None, :] - Gam)
    dGam -= dKh * Kh
    dGamC = dGamC + np.sum(dKh * Kh, axis=0)
    dGam[-1] += dGamC
    extras = dict(d_delta=d_delta, dAqk=dAqk, dAkk=dAkk, dKh=dKh, dQt=dQt, dw=dw, dGamC=dGamC)
    return dq, dk, dv, dGam, dbeta, dS_in, extras


def run_chunked(q, k, v, g, beta, scale, h0=None, do=None, dht=None, cu_seqlens=None, *, chunk=64,
                keep=False):
    """Chunk-parallel forward + backward with the same interface and outputs
    as :func:`oracle.run` (plus s_in / ds_out). With ``keep`` the per-chunk
    intermediates are returned under ``"chunks"`` keyed by (global chunk, hv).
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    h0, do, dht = _f64(h0), _f64(do), _f64(dht)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    G = HV // H
    if cu_seqlens is None:
        cu = [b * T for b in range(B + 1)]
    else:
        cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    N = len(cu) - 1
    qf, kf = q.reshape(-1, H, K), k.reshape(-1, H, K)
    vf, gf, bf = v.reshape(-1, HV, V), g.reshape(-1, HV, K), beta.reshape(-1, HV)
    dof = do.reshape(-1, HV, V) if do is not None else np.zeros_like(vf)
    R = qf.shape[0]
    o = np.zeros((R, HV, V))
    dq, dk = np.zeros((R, H, K)), np.zeros((R, H, K))
    dv, dg, db = np.zeros((R, HV, V)), np.zeros((R, HV, K)), np.zeros((R, HV))
    ht, dh0 = np.zeros((N, HV, K, V)), np.zeros((N, HV, K, V))
    choff = [0]
    for n in range(N):
        choff.append(choff[-1] + -(-(cu[n + 1] - cu[n]) // chunk))
    s_in_all = np.zeros((choff[-1], HV, K, V))
    ds_out_all = np.zeros((choff[-1], HV, K, V))
    chunks = {}
    for n in range(N):
        bos, eos = cu[n], cu[n + 1]
        nt = choff[n + 1] - choff[n]
        for hv in range(HV):
            h = hv // G
            S = h0[n, hv].copy() if h0 is not None else np.zeros((K, V))
            fw = []
            for i in range(nt):
                r0, r1 = bos + i * chunk, min(eos, bos + (i + 1) * chunk)
                f = chunk_forward(qf[r0:r1, h], kf[r0:r1, h], vf[r0:r1, hv], gf[r0:r1, hv], bf[r0:r1, hv],
                                  scale, S)
                o[r0:r1, hv] = f["O"]
                s_in_all[choff[n] + i, hv] = S
                S = f["S_out"]
                fw.append(f)
            ht[n, hv] = S
            dS = dht[n, hv].copy() if dht is not None else np.zeros((K, V))
            for i in reversed(range(nt)):
                r0, r1 = bos + i * chunk, min(eos, bos + (i + 1) * chunk)
                ds_out_all[choff[n] + i, hv] = dS
                dqc, dkc, dvc, dGam, dbc, dS, ex = chunk_backward(
                    fw[i], qf[r0:r1, h], kf[r0:r1, h], vf[r0:r1, hv], bf[r0:r1, hv], scale, dof[r0:r1, hv], dS)
                dq[r0:r1, h] += dqc
                dk[r0:r1, h] += dkc
                dv[r0:r1, hv] = dvc
                db[r0:r1, hv] = dbc
                dg[r0:r1, hv] = np.cumsum(dGam[::-1], axis=0)[::-1]
                if keep:
                    chunks[(choff[n] + i, hv)] = dict(fw[i], **ex, dS_out=ds_out_all[choff[n] + i, hv])
            dh0[n, hv] = dS
    out = dict(o=o.reshape(B, T, HV, V), ht=ht, dq=dq.reshape(B, T, H, K), dk=dk.reshape(B, T, H, K),
               dv=dv.reshape(B, T, HV, V), dg=dg.reshape(B, T, HV, K), dbeta=db.reshape(B, T, HV), dh0=dh0,
               s_in=s_in_all, ds_out=ds_out_all)
    if keep:
        out["chunks"] = chunks
    return out
