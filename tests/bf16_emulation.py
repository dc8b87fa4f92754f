"""A numpy model of the bf16 tensor-core path's rounding, for one (sequence, head) unit.

Test infrastructure: it restates, in fp64, the chunkwise algebra the bf16 kernels
evaluate (the UT/WY form per 64-token chunk, the state carried across chunks, and the
chain rule back through the same steps), and rounds to bf16 exactly the intermediates
the kernels hold as bf16 tensor-core operands or workspace images.  Every rounding
point can be switched off (exact), kept (bf16, as the kernels do) or replaced by a
two-term bf16 split (hi + lo, about 16 mantissa bits).  It shares nothing with the
CUDA library; the fp64 oracle is its reference.  Used by tests/test_bf16_precision.py
to show which precision the absolute error bound would need.

Notation (per chunk, Gamma the within-chunk cumulative log-decay per key channel):
  Kb = k e^Gamma, Kr = k e^-Gamma, Qb = q e^Gamma, KC = k e^{Gamma_last - Gamma}
  T = (I + diag(beta) strict_lower(Kb Kr^T))^-1, Wy = T diag(beta) Kb, Ut = T diag(beta) v
  Aqk = tril(Qb Kr^T), Qt = s (Qb - Aqk Wy), Ot = s Aqk Ut
  U = Ut - Wy S, O = Qt S + Ot, S' = diag(e^{Gamma_last}) S + KC^T U
"""
from __future__ import annotations

import numpy as np
import torch

# the bf16 rounding points of the kernels, in the order the data flows
FORWARD_POINTS = ("Qb", "Kr", "Kb", "bKb", "bV", "KC", "T", "Wy", "Ut", "Aqk", "Qt", "Ot",
                  "S", "U", "S_img", "U_img")
BACKWARD_POINTS = ("dS", "dU", "dS_img", "dQt", "dWyA", "P", "dAqk", "dWy", "dUt", "dT", "X",
                   "dG")
ALL_POINTS = FORWARD_POINTS + BACKWARD_POINTS
# the operands that carry the state across chunks and the UT inverse
STATE_POINTS = ("S", "dS", "U", "dU", "T", "S_img", "dS_img", "U_img")


def bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


class Rounding:
    """bf16 at the points in `bf`, a hi + lo bf16 pair at the points in `split`,
    exact elsewhere."""

    def __init__(self, bf=(), split=()):
        self.bf, self.split = set(bf), set(split)

    def __call__(self, name: str, x: np.ndarray) -> np.ndarray:
        if name in self.split:
            hi = bf16(x)
            return hi + bf16(x - hi)
        if name in self.bf:
            return bf16(x)
        return x


def run_unit(rnd, variant, q, k, v, beta, g, h0, dO, dhT, scale=1.0, C=64):
    """Forward and backward of one unit: q, k, v, dO [T, d]; beta [T]; g [T] (Gated
    DeltaNet), [T, d] (KDA) or None; h0, dhT [d, d] or None.  Returns o, hT and the
    gradient dict (dq, dk, dv, dbeta, dg, dh0)."""
    T, D = q.shape
    S = np.zeros((D, D)) if h0 is None else h0.copy()
    o = np.zeros((T, D))
    saved = []
    for a in range(0, T, C):
        b = min(T, a + C)
        L = b - a
        if variant == "deltanet":
            G = np.zeros((L, D))
        elif variant == "gdn":
            G = np.repeat(np.cumsum(g[a:b])[:, None], D, axis=1)
        else:
            G = np.cumsum(g[a:b], axis=0)
        e, ei, eL = np.exp(G), np.exp(-G), np.exp(G[-1])
        qq, kk, vv, bb = q[a:b], k[a:b], v[a:b], beta[a:b]
        Qb, Kr, Kb = rnd("Qb", qq * e), rnd("Kr", kk * ei), rnd("Kb", kk * e)
        bKb, bV = rnd("bKb", bb[:, None] * kk * e), rnd("bV", bb[:, None] * vv)
        KC = rnd("KC", kk * eL[None, :] * ei)
        Gram = Kb @ Kr.T
        Tm = rnd("T", np.linalg.inv(np.eye(L) + bb[:, None] * np.tril(Gram, -1)))
        Wy, Ut = rnd("Wy", Tm @ bKb), rnd("Ut", Tm @ bV)
        Aqk = rnd("Aqk", np.tril(Qb @ Kr.T))
        Qt = rnd("Qt", scale * (Qb - Aqk @ Wy))
        Ot = rnd("Ot", scale * Aqk @ Ut)
        Sb = rnd("S", S)
        U = rnd("U", Ut - Wy @ Sb)
        o[a:b] = Ot + Qt @ Sb
        saved.append(dict(a=a, b=b, e=e, ei=ei, eL=eL, Qb=Qb, Kr=Kr, Kb=Kb, KC=KC, T=Tm, Wy=Wy,
                          Qt=Qt, S=rnd("S_img", S), U=rnd("U_img", U)))
        S = eL[:, None] * S + KC.T @ U
    hT = S
    dS = np.zeros((D, D)) if dhT is None else dhT.copy()
    dq, dk, dv = np.zeros((T, D)), np.zeros((T, D)), np.zeros((T, D))
    dbeta, dgam = np.zeros(T), np.zeros((T, D))
    for r in reversed(saved):
        a, b = r["a"], r["b"]
        L = b - a
        kk, vv, bb, dOc = k[a:b], v[a:b], beta[a:b], dO[a:b]
        Qb, Kr, Kb, e, ei, eL, Tm = r["Qb"], r["Kr"], r["Kb"], r["e"], r["ei"], r["eL"], r["T"]
        # the backward scan
        dU = rnd("dU", r["KC"] @ rnd("dS", dS))
        dS_img = rnd("dS_img", dS)
        dS_prev = eL[:, None] * dS + r["Qt"].T @ dOc - r["Wy"].T @ dU
        # the chunk's gradients from the stored images
        dQt = rnd("dQt", dOc @ r["S"].T)
        mdWyA = rnd("dWyA", -dU @ r["S"].T)
        dKC = r["U"] @ dS_img.T
        dgC = np.sum(dS_img * r["S"], axis=1)
        Aqk = rnd("Aqk", np.tril(Qb @ Kr.T))
        P = rnd("P", bb[None, :] * (dOc @ vv.T - dQt @ Kb.T))
        dAqk = rnd("dAqk", scale * np.tril(P @ Tm.T))
        dWy = rnd("dWy", mdWyA - scale * Aqk.T @ dQt)
        dUt = rnd("dUt", dU + scale * Aqk.T @ dOc)
        M = dWy @ Kb.T + dUt @ vv.T
        db = np.sum(Tm * M, axis=0)
        dT = rnd("dT", M * bb[None, :])
        dbV, dbK = Tm.T @ dUt, Tm.T @ dWy
        X = rnd("X", dT @ Tm.T)
        dA = -np.tril(Tm.T @ X, -1)
        db = db + np.sum(dA * (Kb @ Kr.T), axis=1)
        dG = rnd("dG", bb[:, None] * dA)
        dQb = scale * dQt + dAqk @ Kr
        dKb = dG @ Kr + bb[:, None] * dbK
        dKr = dG.T @ Kb + dAqk.T @ Qb
        dq[a:b] = dQb * e
        dk[a:b] = dKb * e + (dKr + dKC * eL[None, :]) * ei
        dv[a:b] = bb[:, None] * dbV
        dbeta[a:b] = db
        dGam = dQb * Qb + dKb * Kb - dKr * Kr - dKC * r["KC"]
        dGam[L - 1] += np.sum(dKC * r["KC"], axis=0) + dgC * eL
        dgam[a:b] = np.cumsum(dGam[::-1], axis=0)[::-1]
        dS = dS_prev
    dg = None if variant == "deltanet" else (dgam.sum(axis=1) if variant == "gdn" else dgam)
    return o, hT, dict(dq=dq, dk=dk, dv=dv, dbeta=dbeta, dg=dg, dh0=dS)
