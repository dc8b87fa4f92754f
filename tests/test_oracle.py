"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test is a different route to a result the recurrence fixes (page "Linear
Attention Architectures: Mechanisms, Trade-offs, and Cross-Layer Routing",
section "Metodologia y Marco de Trabajo", item 1: decay before the residual,
residual r = v - vbar, write of the residual; the three variant bullets):

* explicit unrolling: the whole sequence solved as one dense lower-triangular
  system (a matrix derivation of the recurrence, numpy fp64 solve);
* central finite differences of the forward for every input;
* symbolic differentiation (sympy, exact rationals) on a tiny case;
* closed forms: beta = 0 (the memory only decays), exact recall of a unit key
  written with beta = 1, orthonormal keys (no interference), a hand-worked
  scalar example stored in tests/golden;
* invariants: DeltaNet == Gated DeltaNet(alpha = 1) == KDA(alpha vector = 1),
  KDA with a channel-constant gate == Gated DeltaNet, chaining two calls through
  the state == one call, packed ragged sequences == separate calls.

A plausible mistake in the oracle (decay after the residual, read before the
write, a transposed state, a sign or a dropped term in the backward) fails at
least one of these.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(variant, B=2, T=13, H=2, dk=5, dv=4, seed=1, h0=True, gscale=0.3,
                unit_keys=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, H, dk))
    k = r.standard_normal((B, T, H, dk))
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, H, dv))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, H))))
    g = None
    if variant == "gdn":
        g = -gscale * np.log1p(np.exp(r.standard_normal((B, T, H))))
    elif variant == "kda":
        g = -gscale * np.log1p(np.exp(r.standard_normal((B, T, H, dk))))
    s0 = 0.3 * r.standard_normal((B, H, dk, dv)) if h0 else None
    dO = r.standard_normal((B, T, H, dv))
    dhT = r.standard_normal((B, H, dk, dv))
    return dict(q=q, k=k, v=v, beta=beta, g=g, h0=s0, dO=dO, dhT=dhT)


def gate_per_channel(variant, g, dk):
    """log-decay per (token, channel) for one sequence/head: [T, dk]."""
    if variant == "deltanet":
        return None
    if variant == "gdn":
        return np.repeat(g[:, None], dk, axis=1)
    return g


def unrolled(variant, q, k, v, beta, g, S0, scale):
    """One sequence, one head.  The recurrence written as one linear system.

    With Gamma_t = sum_{s<=t} log a_s (per key channel) and u_t = beta_t r_t:
      S_t = diag(e^{Gamma_t}) S_0 + sum_{j<=t} diag(e^{Gamma_t - Gamma_j}) k_j u_j^T
    and the residual against the decayed memory gives
      (I + diag(beta) strict_lower(Kbar Kbrev^T)) U = diag(beta) (V - Kbar S_0),
    Kbar = K * e^{Gamma}, Kbrev = K * e^{-Gamma};  O = scale (Qbar S_0 +
    tril(Qbar Kbrev^T) U);  S_T = diag(e^{Gamma_T}) S_0 + (K * e^{Gamma_T - Gamma})^T U.
    """
    T, dk = k.shape
    G = np.zeros((T, dk)) if g is None else np.cumsum(g, axis=0)
    Kb = k * np.exp(G)
    Kr = k * np.exp(-G)
    Qb = q * np.exp(G)
    M = np.eye(T) + np.diag(beta) @ np.tril(Kb @ Kr.T, -1)
    U = np.linalg.solve(M, np.diag(beta) @ (v - Kb @ S0))
    O = scale * (Qb @ S0 + np.tril(Qb @ Kr.T) @ U)
    ST = np.exp(G[-1])[:, None] * S0 + (k * np.exp(G[-1] - G)).T @ U
    return O, ST, U


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
@pytest.mark.parametrize("scale", [1.0, 0.7])
def test_forward_matches_unrolled_solve(variant, scale):
    x = rand_inputs(variant, B=2, T=13, H=2, dk=5, dv=4)
    o, hT, u = oracle.forward(variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                              scale=scale, want_u=True)
    for b in range(2):
        for h in range(2):
            g = gate_per_channel(variant, None if x["g"] is None else x["g"][b, :, h],
                                 5)
            O, ST, U = unrolled(variant, x["q"][b, :, h], x["k"][b, :, h], x["v"][b, :, h],
                                x["beta"][b, :, h], g, x["h0"][b, h], scale)
            np.testing.assert_allclose(o[b, :, h], O, rtol=0, atol=1e-12)
            np.testing.assert_allclose(hT[b, h], ST, rtol=0, atol=1e-12)
            # the emitted write u_t = beta_t r_t is the unknown of the unrolled system
            np.testing.assert_allclose(u[b, :, h], U, rtol=0, atol=1e-12)


def loss_of(variant, x, scale=1.0, **kw):
    o, hT = oracle.forward(variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                           scale=scale, **kw)
    return float(np.sum(o * x["dO"]) + np.sum(hT * x["dhT"]))


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
def test_backward_matches_central_differences(variant):
    scale = 0.9
    x = rand_inputs(variant, B=2, T=9, H=2, dk=3, dv=2, seed=7)
    grads = oracle.backward(variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                            x["dO"], x["dhT"], scale=scale)
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("h0", "dh0")]
    if variant != "deltanet":
        names.append(("g", "dg"))
    h = 1e-6
    for name, gname in names:
        base = x[name]
        fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = dict(x)
            xp[name] = base.copy()
            xp[name][idx] += h
            lp = loss_of(variant, xp, scale)
            xp[name][idx] -= 2 * h
            lm = loss_of(variant, xp, scale)
            fd[idx] = (lp - lm) / (2 * h)
        an = grads[gname]
        err = np.max(np.abs(an - fd)) / max(1.0, np.max(np.abs(fd)))
        assert err < 1e-6, f"{variant} {gname}: relative error {err}"


def loss_with_write(variant, x, scale):
    o, hT, u = oracle.forward(variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                              scale=scale, want_u=True)
    return float(np.sum(o * x["dO"]) + np.sum(hT * x["dhT"]) + np.sum(u * x["dU"]))


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
def test_write_gradient_matches_central_differences(variant):
    """L = sum(dO o) + sum(dhT hT) + sum(dU u) with u the emitted write beta r."""
    scale = 0.8
    x = rand_inputs(variant, B=1, T=8, H=2, dk=3, dv=2, seed=17)
    x["dU"] = np.random.default_rng(18).standard_normal(x["v"].shape)
    grads = oracle.backward(variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                            x["dO"], x["dhT"], scale=scale, dU=x["dU"])
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("h0", "dh0")]
    if variant != "deltanet":
        names.append(("g", "dg"))
    h = 1e-6
    for name, gname in names:
        base = x[name]
        fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = dict(x)
            xp[name] = base.copy()
            xp[name][idx] += h
            lp = loss_with_write(variant, xp, scale)
            xp[name][idx] -= 2 * h
            lm = loss_with_write(variant, xp, scale)
            fd[idx] = (lp - lm) / (2 * h)
        an = grads[gname]
        err = np.max(np.abs(an - fd)) / max(1.0, np.max(np.abs(fd)))
        assert err < 1e-6, f"{variant} {gname}: relative error {err}"


def test_write_gradient_closed_form_last_token():
    """With only dU in the loss, the last token's value reaches nothing but its own
    write u_T = beta_T (v_T - Wd_T k_T): dv_T = beta_T dU_T exactly, and dbeta_T =
    r_T . dU_T = u_T . dU_T / beta_T."""
    x = rand_inputs("kda", B=2, T=6, H=2, dk=4, dv=3, seed=19)
    dU = np.random.default_rng(20).standard_normal(x["v"].shape)
    zero = np.zeros_like(x["dO"])
    _, _, u = oracle.forward("kda", x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                             want_u=True)
    gr = oracle.backward("kda", x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], zero,
                         None, dU=dU)
    b = x["beta"][:, -1, :, None]
    np.testing.assert_allclose(gr["dv"][:, -1], b * dU[:, -1], rtol=0, atol=1e-13)
    np.testing.assert_allclose(gr["dbeta"][:, -1],
                               np.sum(u[:, -1] * dU[:, -1], axis=-1) / x["beta"][:, -1],
                               rtol=1e-12, atol=1e-13)


def test_backward_matches_symbolic_gradient():
    """Exact derivatives by sympy on a tiny KDA case (T=3, dk=2, dv=2), with
    rational inputs; the symbolic forward is built from the four lines of the
    recurrence, the gradient by sympy's own differentiation."""
    sp = pytest.importorskip("sympy")
    T, dk, dv = 3, 2, 2
    rng = np.random.default_rng(3)

    qn = rng.standard_normal((T, dk)); kn = rng.standard_normal((T, dk))
    vn = rng.standard_normal((T, dv)); bn = np.array([0.5, 0.25, 0.75])
    gn = -np.abs(rng.standard_normal((T, dk))) * 0.5
    s0n = rng.standard_normal((dk, dv)) * 0.5
    dOn = rng.standard_normal((T, dv))
    # quantise to multiples of 1/64 so sympy and the oracle see identical values
    qn, kn, vn, gn, s0n, dOn = [np.round(a * 64) / 64 for a in (qn, kn, vn, gn, s0n, dOn)]
    syms = {}

    def symmat(name, shape):
        m = sp.Matrix(shape[0], shape[1], lambda i, j: sp.Symbol(f"{name}_{i}_{j}"))
        syms[name] = m
        return m

    Q = symmat("q", (T, dk)); K = symmat("k", (T, dk)); V = symmat("v", (T, dv))
    Bt = symmat("b", (T, 1)); Gs = symmat("g", (T, dk)); S0 = symmat("s", (dk, dv))
    W = S0.T  # d_v x d_k
    loss = 0
    for t in range(T):
        D = sp.diag(*[sp.exp(Gs[t, c]) for c in range(dk)])
        Wd = W * D
        r = V[t, :].T - Wd * K[t, :].T
        W = Wd + Bt[t, 0] * r * K[t, :]
        o = W * Q[t, :].T
        loss += sum(o[j] * sp.Rational(int(round(dOn[t, j] * 64)), 64) for j in range(dv))
    vals = {}
    for name, arr in (("q", qn), ("k", kn), ("v", vn), ("b", bn[:, None]), ("g", gn),
                      ("s", s0n)):
        m = syms[name]
        for i in range(m.rows):
            for j in range(m.cols):
                vals[m[i, j]] = sp.Rational(int(round(arr[i, j] * 64)), 64)
    grads = oracle.backward("kda", qn[None, :, None], kn[None, :, None], vn[None, :, None],
                            bn[None, :, None], gn[None, :, None], s0n[None, None],
                            dOn[None, :, None], None)
    table = (("q", grads["dq"][0, :, 0]), ("k", grads["dk"][0, :, 0]),
             ("v", grads["dv"][0, :, 0]), ("b", grads["dbeta"][0, :, 0][:, None]),
             ("g", grads["dg"][0, :, 0]), ("s", grads["dh0"][0, 0]))
    for name, got in table:
        m = syms[name]
        for i in range(m.rows):
            for j in range(m.cols):
                exact = float(sp.diff(loss, m[i, j]).subs(vals).evalf(30))
                assert abs(got[i, j] - exact) < 1e-12 * max(1.0, abs(exact)), (name, i, j)


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
def test_beta_zero_closed_form(variant):
    """beta = 0: nothing is written, the memory only decays:
    S_t = diag(prod a) S_0, o_t = scale S_t^T q_t, and dk = dv = 0 exactly."""
    x = rand_inputs(variant, B=1, T=10, H=2, dk=4, dv=3, seed=11)
    x["beta"] = np.zeros_like(x["beta"])
    o, hT = oracle.forward(variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                           scale=1.3)
    for h in range(2):
        g = gate_per_channel(variant, None if x["g"] is None else x["g"][0, :, h], 4)
        G = np.zeros((10, 4)) if g is None else np.cumsum(g, axis=0)
        S0 = x["h0"][0, h]
        for t in range(10):
            St = np.exp(G[t])[:, None] * S0
            np.testing.assert_allclose(o[0, t, h], 1.3 * St.T @ x["q"][0, t, h], atol=1e-13)
        np.testing.assert_allclose(hT[0, h], np.exp(G[-1])[:, None] * S0, atol=1e-13)
    gr = oracle.backward(variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                         x["dO"], x["dhT"], scale=1.3)
    assert np.all(gr["dk"] == 0.0) and np.all(gr["dv"] == 0.0)
    assert np.any(gr["dbeta"] != 0.0)


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
def test_exact_recall(variant):
    """A unit-norm key written with beta = 1 and read back with q = k returns
    its value exactly, whatever the prior state and the decay."""
    x = rand_inputs(variant, B=2, T=11, H=2, dk=6, dv=5, seed=5)
    x["beta"] = np.ones_like(x["beta"])
    x["q"] = x["k"].copy()
    o, _ = oracle.forward(variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"])
    np.testing.assert_allclose(o, x["v"], atol=1e-13)


def test_variant_nesting():
    x = rand_inputs("kda", B=2, T=17, H=2, dk=4, dv=3, seed=9)
    a = dict(q=x["q"], k=x["k"], v=x["v"], beta=x["beta"], h0=x["h0"])
    o_dn, s_dn = oracle.forward("deltanet", **a)
    g_gdn0 = np.zeros(x["beta"].shape)
    g_kda0 = np.zeros(x["q"].shape)
    o_g, s_g = oracle.forward("gdn", g=g_gdn0, **a)
    o_k, s_k = oracle.forward("kda", g=g_kda0, **a)
    assert np.array_equal(o_dn, o_g) and np.array_equal(s_dn, s_g)
    assert np.array_equal(o_dn, o_k) and np.array_equal(s_dn, s_k)
    # a gate that is constant across channels makes KDA equal to Gated DeltaNet
    gs = -0.2 * np.log1p(np.exp(np.random.default_rng(2).standard_normal(x["beta"].shape)))
    gv = np.repeat(gs[..., None], 4, axis=-1)
    o_g, s_g = oracle.forward("gdn", g=gs, **a)
    o_k, s_k = oracle.forward("kda", g=gv, **a)
    np.testing.assert_allclose(o_g, o_k, atol=1e-14)
    np.testing.assert_allclose(s_g, s_k, atol=1e-14)
    gg = oracle.backward("gdn", g=gs, dO=x["dO"], dhT=x["dhT"], **a)
    gk = oracle.backward("kda", g=gv, dO=x["dO"], dhT=x["dhT"], **a)
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(gg[n], gk[n], atol=1e-13)
    np.testing.assert_allclose(gg["dg"], gk["dg"].sum(-1), atol=1e-13)
    gd = oracle.backward("deltanet", dO=x["dO"], dhT=x["dhT"], g=None, **a)
    g0 = oracle.backward("gdn", g=g_gdn0, dO=x["dO"], dhT=x["dhT"], **a)
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        assert np.array_equal(gd[n], g0[n])


def test_orthonormal_keys_store_without_interference():
    """DeltaNet from W0 = 0 with orthonormal keys: every residual is the full
    value, so W_T = sum_t beta_t v_t k_t^T (plain linear attention)."""
    rng = np.random.default_rng(4)
    dk, dv, T = 8, 3, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm[:, :T].T.copy()
    v = rng.standard_normal((T, dv))
    beta = rng.uniform(0.1, 0.9, T)
    q = rng.standard_normal((T, dk))
    o, hT = oracle.forward("deltanet", q[None, :, None], k[None, :, None], v[None, :, None],
                           beta[None, :, None])
    S = sum(beta[t] * np.outer(k[t], v[t]) for t in range(T))
    np.testing.assert_allclose(hT[0, 0], S, atol=1e-14)
    for t in range(T):
        St = sum(beta[s] * np.outer(k[s], v[s]) for s in range(t + 1))
        np.testing.assert_allclose(o[0, t, 0], St.T @ q[t], atol=1e-14)


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rhs = line.split("=", 1)
            vals[key.strip()] = [float(s) for s in rhs.split()]
    return vals


def test_hand_worked_scalar_example():
    gv = read_golden("scalar_gdn_t2.txt")
    q = np.array(gv["q"]).reshape(1, 2, 1, 1)
    k = np.array(gv["k"]).reshape(1, 2, 1, 1)
    v = np.array(gv["v"]).reshape(1, 2, 1, 1)
    beta = np.array(gv["beta"]).reshape(1, 2, 1)
    g = np.log(np.array(gv["alpha"])).reshape(1, 2, 1)
    h0 = np.array(gv["W0"]).reshape(1, 1, 1, 1)
    o, hT = oracle.forward("gdn", q, k, v, beta, g, h0)
    np.testing.assert_allclose(o.ravel(), gv["o"], atol=1e-14)
    np.testing.assert_allclose(hT.ravel(), gv["WT"], atol=1e-14)
    gr = oracle.backward("gdn", q, k, v, beta, g, h0, np.ones_like(o), None)
    for key, name in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dbeta", "dbeta"),
                      ("dW0", "dh0"), ("dg", "dg")):
        np.testing.assert_allclose(gr[name].ravel(), gv[key], atol=1e-14, err_msg=key)


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
def test_split_and_packed_consistency(variant):
    x = rand_inputs(variant, B=1, T=150, H=2, dk=4, dv=3, seed=12)
    a = {n: x[n] for n in ("q", "k", "v", "beta", "g")}

    def cut(d, lo, hi):
        return {n: (None if val is None else val[:, lo:hi]) for n, val in d.items()}

    o, hT = oracle.forward(variant, h0=x["h0"], **a)
    o1, h1 = oracle.forward(variant, h0=x["h0"], **cut(a, 0, 70))
    o2, h2 = oracle.forward(variant, h0=h1, **cut(a, 70, 150))
    assert np.array_equal(np.concatenate([o1, o2], 1), o) and np.array_equal(h2, hT)
    gr = oracle.backward(variant, h0=x["h0"], dO=x["dO"], dhT=x["dhT"], **a)
    g2 = oracle.backward(variant, h0=h1, dO=x["dO"][:, 70:], dhT=x["dhT"],
                         **cut(a, 70, 150))
    g1 = oracle.backward(variant, h0=x["h0"], dO=x["dO"][:, :70], dhT=g2["dh0"],
                         **cut(a, 0, 70))
    for n in ("dq", "dk", "dv", "dbeta") + (("dg",) if variant != "deltanet" else ()):
        np.testing.assert_allclose(np.concatenate([g1[n], g2[n]], 1), gr[n], atol=1e-12)
    np.testing.assert_allclose(g1["dh0"], gr["dh0"], atol=1e-12)

    # packed ragged sequences (with an empty one) == separate calls
    lens = [40, 0, 65, 45]
    cu = np.cumsum([0] + lens).astype(np.int32)
    N = len(lens)
    rng = np.random.default_rng(13)
    h0s = rng.standard_normal((N, 2, 4, 3)) * 0.1
    dhTs = rng.standard_normal((N, 2, 4, 3))
    op, hp = oracle.forward(variant, h0=h0s, cu_seqlens=cu, **a)
    gp = oracle.backward(variant, h0=h0s, dO=x["dO"], dhT=dhTs, cu_seqlens=cu, **a)
    for n in range(N):
        lo, hi = cu[n], cu[n + 1]
        on, hn = oracle.forward(variant, h0=h0s[n:n + 1], **cut(a, lo, hi))
        assert np.array_equal(op[:, lo:hi], on) and np.array_equal(hp[n:n + 1], hn)
        gn = oracle.backward(variant, h0=h0s[n:n + 1], dO=x["dO"][:, lo:hi],
                             dhT=dhTs[n:n + 1], **cut(a, lo, hi))
        for m in ("dq", "dk", "dv", "dbeta") + (("dg",) if variant != "deltanet" else ()):
            assert np.array_equal(gp[m][:, lo:hi], gn[m])
        assert np.array_equal(gp["dh0"][n:n + 1], gn["dh0"])
    assert np.array_equal(hp[1], h0s[1]) and np.array_equal(gp["dh0"][1], dhTs[1])


def test_units_subset_matches_full_run():
    x = rand_inputs("kda", B=2, T=30, H=3, dk=4, dv=3, seed=21)
    a = {n: x[n] for n in ("q", "k", "v", "beta", "g", "h0")}
    o, hT = oracle.forward("kda", **a)
    units = np.array([4, 1], dtype=np.int32)   # (seq 1, head 1), (seq 0, head 1)
    os_, hs = oracle.forward("kda", units=units, **a)
    for u in units:
        n, h = divmod(int(u), 3)
        assert np.array_equal(os_[n, :, h], o[n, :, h])
        assert np.array_equal(hs[n, h], hT[n, h])
    assert np.all(os_[0, :, 0] == 0)
