"""Reverse mode of the KDA forward in its chunked WY form, fp64 numpy.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the product path never
imports it.

What it computes: the same gradients as :func:`oracle.bwd` (the token-level
reverse mode in ``kda_oracle.c``), but block by block in the chunked form of the
forward that "feat(kda): SM90 FlashKDA prefill, intracard CP, and backend
dispatch" (commit notes: K1 prepares decayed q/k, beta and the WY inverse; K2
runs the inter-chunk recurrence) computes, which is the form a chunked,
tensor-core backward evaluates.  The pages' kernels are forward only, so the
steps below are this build's derivation; they are written once here, in the
notation of the forward, and pinned against the token-level reverse mode (itself
pinned by central differences of the forward) in ``tests/test_oracle_bwd_pins.py``.

Forward of one block of C tokens from its start state S (K x V), with
Gam_t = exp(sum_{s<=t} log alpha_s) per channel inside the block, hats for the
l2-normalised rows and the token recurrence's u_t as the rows of U:
    Kt = K^ o Gam,  Kb = K^ / Gam,  Qt = Q^ o Gam              (C x K)
    A  = strict_lower(Diag(beta) Kt Kb^T),  T = (I + A)^-1        (C x C)
    W  = T Diag(beta) Kt,  U~ = T Diag(beta) V,  U = U~ - W S     (C x K, C x V)
    M  = lower_incl(Qt Kb^T)
    O  = scale (Qt S + M U)
    S' = Diag(Gam_C) (S + Kb^T U)
Reverse, given dO and dS' (G = Diag(Gam_C) dS'):
    dS  = G + scale Qt^T dO - W^T dU
    dU  = Kb G + scale M^T dO                      dU~ = dU,  dW = -dU S^T
    dKb = U G^T + dM^T Qt + dP^T Kt              dM = scale lower_incl(dO U^T)
    dQt = scale dO S^T + dM Kb
    dT  = dW (Diag(beta) Kt)^T + dU~ (Diag(beta) V)^T
    dA  = strict_lower(-T^T dT T^T),   dP = Diag(beta) dA   (P = Kt Kb^T)
    dKt = Diag(beta) T^T dW + dP Kb
    dV  = Diag(beta) T^T dU~
    dbeta = rowsum(V o T^T dU~) + rowsum(Kt o T^T dW) + rowsum(dA o P)
    dK^ = dKt o Gam + dKb / Gam,   dQ^ = dQt o Gam
    dlg_t = dKt o Kt - dKb o Kb + dQt o Qt  (+ Gam_C o rowsum_v((S + Kb^T U) o dS') at t = C-1)
    dlog alpha_s = sum_{t >= s} dlg_t
then the preprocessing's reverse, as in the token-level form: the l2 norms, the
gate log alpha = lower_bound sigmoid(exp(A_log)(g + dt_bias)) and beta = sigmoid.
"""
from __future__ import annotations

import numpy as np

from . import KD, _as_f64


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def _unit(q, k, v, pre, braw, lb, scale, S0, dO, dSf, C):
    """One (sequence, value head): rows [T, 128]; S0, dSf as K x V.  Returns the
    gradients with respect to q, k, v, the gate pre-activation, the beta logits and
    the initial state (K x V)."""
    T = q.shape[0]
    rq = 1.0 / np.sqrt((q * q).sum(1) + 1e-6)
    rk = 1.0 / np.sqrt((k * k).sum(1) + 1e-6)
    qh, kh = q * rq[:, None], k * rk[:, None]
    beta = _sig(braw)
    la = lb * _sig(pre)                                   # log alpha, [T, K]
    # forward sweep: block start states and u_t (the rows of U)
    S = S0.copy()
    starts, U_all = [], np.zeros_like(v)
    for t in range(T):
        if t % C == 0:
            starts.append(S.copy())
        S = np.exp(la[t])[:, None] * S
        u = beta[t] * (v[t] - S.T @ kh[t])
        S = S + np.outer(kh[t], u)
        U_all[t] = u
    dS = dSf.copy()
    dqh, dkh = np.zeros_like(q), np.zeros_like(k)
    dv, dbeta, dla = np.zeros_like(v), np.zeros(T), np.zeros_like(la)
    for b in reversed(range(len(starts))):
        t0, t1 = b * C, min(T, (b + 1) * C)
        n = t1 - t0
        Sc = starts[b]
        Gam = np.exp(np.cumsum(la[t0:t1], axis=0))
        GC = Gam[-1]
        Kh, Qh, V, bt, U = kh[t0:t1], qh[t0:t1], v[t0:t1], beta[t0:t1], U_all[t0:t1]
        Kt, Kb, Qt = Kh * Gam, Kh / Gam, Qh * Gam
        P = Kt @ Kb.T
        Tm = np.linalg.inv(np.eye(n) + np.tril(bt[:, None] * P, -1))
        Bk, Bv = bt[:, None] * Kt, bt[:, None] * V
        W = Tm @ Bk
        M = np.tril(Qt @ Kb.T)
        dOb = dO[t0:t1]
        G = GC[:, None] * dS
        dGC = ((Sc + Kb.T @ U) * dS).sum(1)
        dM = scale * np.tril(dOb @ U.T)
        dU = Kb @ G + scale * (M.T @ dOb)
        dKb = U @ G.T + dM.T @ Qt
        dQt = scale * (dOb @ Sc.T) + dM @ Kb
        dW = -dU @ Sc.T
        dSc = G + scale * (Qt.T @ dOb) - W.T @ dU
        dT = dW @ Bk.T + dU @ Bv.T
        TdW, TdU = Tm.T @ dW, Tm.T @ dU
        dA = np.tril(-Tm.T @ dT @ Tm.T, -1)
        dP = bt[:, None] * dA
        dKt = bt[:, None] * TdW + dP @ Kb
        dKb += dP.T @ Kt
        dv[t0:t1] += bt[:, None] * TdU
        dbeta[t0:t1] += (V * TdU).sum(1) + (Kt * TdW).sum(1) + (dA * P).sum(1)
        dkh[t0:t1] += dKt * Gam + dKb / Gam
        dqh[t0:t1] += dQt * Gam
        dlg = dKt * Kt - dKb * Kb + dQt * Qt
        dlg[-1] += dGC * GC
        dla[t0:t1] += np.cumsum(dlg[::-1], axis=0)[::-1]
        dS = dSc
    dq = rq[:, None] * (dqh - (qh * dqh).sum(1)[:, None] * qh)
    dk = rk[:, None] * (dkh - (kh * dkh).sum(1)[:, None] * kh)
    dpre = dla * lb * _sig(pre) * _sig(-pre)
    dbraw = dbeta * beta * _sig(-braw)
    return dq, dk, dv, dpre, dbraw, dS


def bwd_chunked(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, dout, initial_state=None,
                dfinal_state=None, cu_seqlens=None, chunk=16):
    """Gradients of L = <dout, out> + <dfinal_state, final_state>, as
    :func:`oracle.bwd` returns them (same arguments and shapes; q/k head
    h // (H // HK) serves value head h), computed block by block in the chunked
    form with blocks of `chunk` tokens."""
    qa = _as_f64(q, "q")
    lead = qa.shape[:-2]
    HK = qa.shape[-2]
    H = np.asarray(v).shape[-2]
    G = H // HK
    T_total = int(np.prod(lead))
    if cu_seqlens is None:
        B, T = (lead if len(lead) == 2 else (1, lead[0]))
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    qf = qa.reshape(T_total, HK, KD)
    kf = _as_f64(k, "k").reshape(T_total, HK, KD)
    vf = _as_f64(v, "v").reshape(T_total, H, KD)
    gf = _as_f64(g, "g").reshape(T_total, H, KD)
    bf = _as_f64(beta, "beta").reshape(T_total, H)
    dOf = _as_f64(dout, "dout").reshape(T_total, H, KD)
    Al = _as_f64(A_log, "A_log").reshape(H)
    dtb = _as_f64(dt_bias, "dt_bias").reshape(H, KD)
    S0 = (np.zeros((N, H, KD, KD)) if initial_state is None
          else _as_f64(initial_state, "initial_state").reshape(N, H, KD, KD))
    dSf = (np.zeros((N, H, KD, KD)) if dfinal_state is None
           else _as_f64(dfinal_state, "dfinal_state").reshape(N, H, KD, KD))
    dq, dk = np.zeros((T_total, HK, KD)), np.zeros((T_total, HK, KD))
    dv, dg = np.zeros((T_total, H, KD)), np.zeros((T_total, H, KD))
    dbeta, dA_log, ddt = np.zeros((T_total, H)), np.zeros(H), np.zeros((H, KD))
    dinit = np.zeros((N, H, KD, KD))
    for n in range(N):
        a, b = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            hk = h // G
            ea = np.exp(Al[h])
            if b == a:
                dinit[n, h] = dSf[n, h]
                continue
            pre = ea * (gf[a:b, h] + dtb[h])
            r = _unit(qf[a:b, hk], kf[a:b, hk], vf[a:b, h], pre, bf[a:b, h], float(lower_bound),
                      float(scale), S0[n, h].T, dOf[a:b, h], dSf[n, h].T, int(chunk))
            dq[a:b, hk] += r[0]
            dk[a:b, hk] += r[1]
            dv[a:b, h] = r[2]
            dg[a:b, h] = r[3] * ea
            dbeta[a:b, h] = r[4]
            ddt[h] += (r[3] * ea).sum(0)
            dA_log[h] += (r[3] * pre).sum()
            dinit[n, h] = r[5].T
    return {"dq": dq.reshape(qa.shape), "dk": dk.reshape(qa.shape),
            "dv": dv.reshape(np.asarray(v).shape), "dg": dg.reshape(np.asarray(v).shape),
            "dbeta": dbeta.reshape(np.asarray(beta).shape), "dA_log": dA_log, "ddt_bias": ddt,
            "dinitial_state": dinit}
