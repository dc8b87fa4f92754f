"""Pins of the Gated DeltaNet-2 oracle (oracle/dro2.c) against facts that do not
come from its token loop.

The pages give this variant in words only ("Linear Attention Architectures:
Mechanisms, Trade-offs, and Cross-Layer Routing", section "Metodologia y Marco de
Trabajo", item 1, the Gated DeltaNet-2 bullet: separate per-channel erase and
write gates).  The oracle follows the reading stated in its header; these tests
pin the oracle to that reading, and the reading to the pinned Gated DeltaNet
oracle where the two must agree.  The reading itself is not pinned by the pages.

* reduction to Gated DeltaNet: erase = write = beta (every channel) gives the
  Gated DeltaNet oracle's outputs, and its gradients (dbeta = sum of the erase
  and write gradients);
* explicit unrolling: one (sequence, head) solved as a dense lower-triangular
  system for the predictions p_t, then the outputs as matrix products (numpy);
* central finite differences of every input;
* exact symbolic derivatives (sympy, rational inputs) of the reading's lines;
* closed forms: no erase and no write (the memory only decays); no erase
  (decayed linear attention, a plain sum); erase = write = 1 with unit keys and
  no decay (exact recall of the last value written under a key);
* packed ragged sequences == separate calls;
* a hand-worked two-token example with different erase and write gates
  (tests/golden/scalar_gdn2_t2.txt).
"""
import numpy as np
import pytest

import oracle


def rand2(B=2, T=11, H=2, dk=4, dv=3, seed=1, h0=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, H, dk))
    k = r.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return dict(q=q, k=k, v=r.standard_normal((B, T, H, dv)),
                erase=r.uniform(0.05, 0.95, (B, T, H, dk)),
                write=r.uniform(0.05, 0.95, (B, T, H, dv)),
                g=-0.3 * np.log1p(np.exp(r.standard_normal((B, T, H)))),
                h0=0.3 * r.standard_normal((B, H, dk, dv)) if h0 else None,
                dO=r.standard_normal((B, T, H, dv)), dhT=r.standard_normal((B, H, dk, dv)))


def fwd(x, scale=1.0, **kw):
    return oracle.forward_gdn2(x["q"], x["k"], x["v"], x["erase"], x["write"], x["g"], x["h0"],
                               scale=scale, **kw)


def test_reduces_to_gated_deltanet():
    x = rand2(seed=2)
    r = np.random.default_rng(3)
    beta = r.uniform(0.05, 0.95, x["g"].shape)
    x["erase"] = np.repeat(beta[..., None], x["k"].shape[-1], axis=-1)
    x["write"] = np.repeat(beta[..., None], x["v"].shape[-1], axis=-1)
    o2, h2 = fwd(x, scale=0.8)
    o1, h1 = oracle.forward("gdn", x["q"], x["k"], x["v"], beta, x["g"], x["h0"], scale=0.8)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(h2, h1, rtol=0, atol=1e-12)
    g2 = oracle.backward_gdn2(x["q"], x["k"], x["v"], x["erase"], x["write"], x["g"], x["h0"],
                              x["dO"], x["dhT"], scale=0.8)
    g1 = oracle.backward("gdn", x["q"], x["k"], x["v"], beta, x["g"], x["h0"], x["dO"], x["dhT"],
                         scale=0.8)
    for n in ("dq", "dk", "dv", "dg", "dh0"):
        np.testing.assert_allclose(g2[n], g1[n], rtol=0, atol=1e-11, err_msg=n)
    dbeta = g2["derase"].sum(-1) + g2["dwrite"].sum(-1)
    np.testing.assert_allclose(dbeta, g1["dbeta"], rtol=0, atol=1e-11)


def unrolled(x, b, h, scale):
    """Outputs of one (sequence b, head h) from the whole-sequence matrix form."""
    q, k, v = x["q"][b, :, h], x["k"][b, :, h], x["v"][b, :, h]
    e, w, g = x["erase"][b, :, h], x["write"][b, :, h], x["g"][b, :, h]
    W0 = np.zeros((v.shape[1], k.shape[1])) if x["h0"] is None else x["h0"][b, h].T
    T = len(g)
    G = np.cumsum(g)
    D = np.exp(G[:, None] - G[None, :])          # e^{Gamma_t - Gamma_i}
    Bm = e * k                                    # erase keys
    Vw = w * v                                    # gated values
    Lb = np.tril(D * (k @ Bm.T), -1)              # [t, i] = e^{..} k_t . b_i, i < t
    Lk = np.tril(D * (k @ k.T), -1)
    rhs = np.exp(G)[:, None] * (k @ W0.T) + Lk @ Vw
    P = np.linalg.solve(np.eye(T) + Lb, rhs)      # predictions p_t (rows)
    Aqk = np.tril(D * (q @ k.T))
    Aqb = np.tril(D * (q @ Bm.T))
    O = scale * (np.exp(G)[:, None] * (q @ W0.T) + Aqk @ Vw - Aqb @ P)
    WT = np.exp(G[-1]) * W0 + (np.exp(G[-1] - G)[:, None] * Vw).T @ k \
        - (np.exp(G[-1] - G)[:, None] * P).T @ Bm
    return O, WT.T


def test_matches_unrolled_solve():
    x = rand2(B=2, T=23, H=2, dk=5, dv=4, seed=4)
    o, hT = fwd(x, scale=0.7)
    for b in range(2):
        for h in range(2):
            O, S = unrolled(x, b, h, 0.7)
            np.testing.assert_allclose(o[b, :, h], O, rtol=0, atol=1e-11)
            np.testing.assert_allclose(hT[b, h], S, rtol=0, atol=1e-11)


def loss(x, scale):
    o, hT = fwd(x, scale)
    return float(np.sum(o * x["dO"]) + np.sum(hT * x["dhT"]))


def test_backward_matches_central_differences():
    scale = 0.9
    x = rand2(B=2, T=9, H=2, dk=3, dv=2, seed=7)
    gr = oracle.backward_gdn2(x["q"], x["k"], x["v"], x["erase"], x["write"], x["g"], x["h0"],
                              x["dO"], x["dhT"], scale=scale)
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("erase", "derase"),
                        ("write", "dwrite"), ("g", "dg"), ("h0", "dh0")):
        base = x[name]
        fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = dict(x)
            xp[name] = base.copy()
            xp[name][idx] += h
            lp = loss(xp, scale)
            xp[name][idx] -= 2 * h
            lm = loss(xp, scale)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(gr[gname] - fd)) / max(1.0, np.max(np.abs(fd)))
        assert err < 1e-6, f"{gname}: relative error {err}"


def test_closed_forms():
    x = rand2(B=1, T=12, H=1, dk=4, dv=3, seed=5)
    G = np.cumsum(x["g"][0, :, 0])
    W0 = x["h0"][0, 0].T
    # no erase, no write: o_t = e^{Gamma_t} W0 q_t
    y = dict(x, erase=np.zeros_like(x["erase"]), write=np.zeros_like(x["write"]))
    o, hT = fwd(y)
    np.testing.assert_allclose(o[0, :, 0], np.exp(G)[:, None] * (x["q"][0, :, 0] @ W0.T),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(hT[0, 0], np.exp(G[-1]) * W0.T, rtol=0, atol=1e-12)
    # no erase: W_t = e^{Gamma_t} W0 + sum_{i<=t} e^{Gamma_t - Gamma_i} (w.v)_i k_i^T
    y = dict(x, erase=np.zeros_like(x["erase"]))
    o, _ = fwd(y)
    q, k = x["q"][0, :, 0], x["k"][0, :, 0]
    vw = (x["write"] * x["v"])[0, :, 0]
    for t in range(12):
        Wt = np.exp(G[t]) * W0 + sum(np.exp(G[t] - G[i]) * np.outer(vw[i], k[i])
                                     for i in range(t + 1))
        np.testing.assert_allclose(o[0, t, 0], Wt @ q[t], rtol=0, atol=1e-12)


def test_exact_recall():
    """erase = write = 1, unit keys, no decay: reading with q = k returns the value
    last written under that key, whatever the memory held before."""
    r = np.random.default_rng(6)
    dk, dv, T = 6, 4, 8
    k = r.standard_normal((1, T, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    x = dict(q=k.copy(), k=k, v=r.standard_normal((1, T, 1, dv)),
             erase=np.ones((1, T, 1, dk)), write=np.ones((1, T, 1, dv)),
             g=np.zeros((1, T, 1)), h0=r.standard_normal((1, 1, dk, dv)))
    o, _ = fwd(x)
    np.testing.assert_allclose(o, x["v"], rtol=0, atol=1e-12)


def test_packed_equals_separate():
    x = rand2(B=1, T=30, H=2, dk=4, dv=3, seed=8, h0=False)
    cu = np.array([0, 7, 7, 19, 30], dtype=np.int32)
    r = np.random.default_rng(9)
    h0 = r.standard_normal((4, 2, 4, 3)) * 0.3
    o, hT = oracle.forward_gdn2(x["q"], x["k"], x["v"], x["erase"], x["write"], x["g"], h0,
                                cu_seqlens=cu)
    for n in range(4):
        lo, hi = cu[n], cu[n + 1]
        sl = lambda t: t[:, lo:hi]
        on, hn = oracle.forward_gdn2(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["erase"]),
                                     sl(x["write"]), sl(x["g"]), h0[n:n + 1])
        np.testing.assert_allclose(o[:, lo:hi], on, rtol=0, atol=1e-13)
        np.testing.assert_allclose(hT[n:n + 1], hn, rtol=0, atol=1e-13)


def test_hand_worked_scalar_example():
    """tests/golden/scalar_gdn2_t2.txt: two tokens with d_k = d_v = 1 and different erase
    and write gates, worked by hand (every value an exact binary fraction)."""
    import os
    gv = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "scalar_gdn2_t2.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, rhs = line.split("=", 1)
                gv[key.strip()] = [float(x) for x in rhs.split()]
    sh = (1, 2, 1, 1)
    q, k, v = (np.array(gv[n]).reshape(sh) for n in ("q", "k", "v"))
    e, wr = np.array(gv["erase"]).reshape(sh), np.array(gv["write"]).reshape(sh)
    g = np.log(np.array(gv["alpha"])).reshape(1, 2, 1)
    h0 = np.array(gv["W0"]).reshape(1, 1, 1, 1)
    o, hT = oracle.forward_gdn2(q, k, v, e, wr, g, h0)
    np.testing.assert_allclose(o.ravel(), gv["o"], atol=1e-14)
    np.testing.assert_allclose(hT.ravel(), gv["WT"], atol=1e-14)
    gr = oracle.backward_gdn2(q, k, v, e, wr, g, h0, np.ones_like(o), None)
    for key, name in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("derase", "derase"),
                      ("dwrite", "dwrite"), ("dg", "dg"), ("dW0", "dh0")):
        np.testing.assert_allclose(gr[name].ravel(), gv[key], atol=1e-14, err_msg=key)


def test_backward_matches_symbolic_gradient():
    """Exact derivatives by sympy on a tiny case (T=3, d_k=2, d_v=2) with rational
    inputs: the symbolic forward is built from the lines of the reading (decay,
    prediction, erase, write, read) and differentiated by sympy itself."""
    sp = pytest.importorskip("sympy")
    T, dk, dv = 3, 2, 2
    rng = np.random.default_rng(13)
    q64 = lambda a: np.round(a * 64) / 64  # binary fractions: sympy and the oracle agree
    qn, kn = q64(rng.standard_normal((T, dk))), q64(rng.standard_normal((T, dk)))
    vn, dOn = q64(rng.standard_normal((T, dv))), q64(rng.standard_normal((T, dv)))
    en, wn = q64(rng.uniform(0.1, 0.9, (T, dk))), q64(rng.uniform(0.1, 0.9, (T, dv)))
    gn = q64(-np.abs(rng.standard_normal(T)) * 0.5)
    s0n = q64(rng.standard_normal((dk, dv)) * 0.5)
    syms = {}

    def symmat(name, shape):
        m = sp.Matrix(shape[0], shape[1], lambda i, j: sp.Symbol(f"{name}_{i}_{j}"))
        syms[name] = m
        return m

    Q = symmat("q", (T, dk)); K = symmat("k", (T, dk)); V = symmat("v", (T, dv))
    E = symmat("e", (T, dk)); Wg = symmat("w", (T, dv)); G = symmat("g", (T, 1))
    S0 = symmat("s", (dk, dv))
    W = S0.T  # d_v x d_k
    loss = 0
    for t in range(T):
        Wd = sp.exp(G[t, 0]) * W
        p = Wd * K[t, :].T                                            # prediction
        b = sp.Matrix(1, dk, lambda _, c: E[t, c] * K[t, c])          # erase key
        vw = sp.Matrix(dv, 1, lambda j, _: Wg[t, j] * V[t, j])        # gated value
        W = Wd - p * b + vw * K[t, :]
        o = W * Q[t, :].T
        loss += sum(o[j] * sp.Rational(int(round(dOn[t, j] * 64)), 64) for j in range(dv))
    vals = {}
    for name, arr in (("q", qn), ("k", kn), ("v", vn), ("e", en), ("w", wn),
                      ("g", gn[:, None]), ("s", s0n)):
        m = syms[name]
        for i in range(m.rows):
            for j in range(m.cols):
                vals[m[i, j]] = sp.Rational(int(round(arr[i, j] * 64)), 64)
    sh = lambda a: a[None, :, None]
    gr = oracle.backward_gdn2(sh(qn), sh(kn), sh(vn), sh(en), sh(wn), gn[None, :, None],
                              s0n[None, None], sh(dOn), None)
    table = (("q", gr["dq"][0, :, 0]), ("k", gr["dk"][0, :, 0]), ("v", gr["dv"][0, :, 0]),
             ("e", gr["derase"][0, :, 0]), ("w", gr["dwrite"][0, :, 0]),
             ("g", gr["dg"][0, :, 0][:, None]), ("s", gr["dh0"][0, 0]))
    for name, got in table:
        m = syms[name]
        for i in range(m.rows):
            for j in range(m.cols):
                exact = float(sp.diff(loss, m[i, j]).subs(vals).evalf(30))
                assert abs(got[i, j] - exact) < 1e-12 * max(1.0, abs(exact)), (name, i, j)
