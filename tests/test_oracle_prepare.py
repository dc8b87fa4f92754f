"""Pins of the oracle's input preparation (oracle/prepare.py) against facts that
do not come from its own formulas:

* closed-form values of the maps: sigmoid(0) = 1/2, sigmoid(-b) = 1 - sigmoid(b),
  -softplus(0) = -log 2, -softplus(x) -> -x for large x and -> -e^x for very
  negative x, -softplus(x) = log(sigmoid(-x));
* the normalisation: |q_hat|^2 = s / (s + eps) with s = |q|^2, invariance under
  positive scaling (up to eps), the zero vector mapped to zero;
* central finite differences of the composite loss (preparation, then the
  recurrence) with respect to the raw q, k, b, x: this checks ``chain`` and the
  composition without using the derivative formulas written in it.

A plausible mistake (a missing projection term in the normalisation gradient,
sigmoid' written as beta instead of beta (1 - beta), a sign of the gate chain)
fails the finite differences.
"""
import numpy as np
import pytest

import oracle
from oracle import prepare as prep


def test_sigmoid_closed_forms():
    assert prep.sigmoid(np.array([0.0]))[0] == 0.5
    b = np.linspace(-6, 6, 25)
    np.testing.assert_allclose(prep.sigmoid(-b), 1.0 - prep.sigmoid(b), rtol=0, atol=1e-15)
    # logit(sigmoid(b)) = b
    s = prep.sigmoid(b)
    np.testing.assert_allclose(np.log(s / (1.0 - s)), b, rtol=0, atol=1e-12)


def test_neg_softplus_closed_forms():
    np.testing.assert_allclose(prep.neg_softplus(np.array([0.0])), [-np.log(2.0)], atol=1e-15)
    big = np.array([40.0, 100.0, 700.0])
    np.testing.assert_allclose(prep.neg_softplus(big), -big, rtol=1e-15)
    tiny = np.array([-40.0, -60.0])
    np.testing.assert_allclose(prep.neg_softplus(tiny), -np.exp(tiny), rtol=1e-12)
    x = np.linspace(-8, 8, 33)
    # log alpha = log(sigmoid(-x)): the decay is the sigmoid of -x
    np.testing.assert_allclose(prep.neg_softplus(x), np.log(prep.sigmoid(-x)), rtol=0,
                               atol=1e-14)
    assert np.all(prep.neg_softplus(x) < 0)


def test_normalize_norm_scale_and_zero():
    r = np.random.default_rng(0)
    q = r.standard_normal((4, 7, 3, 16)) * r.uniform(0.1, 10, (4, 7, 3, 1))
    qh = prep.normalize(q)
    s = np.sum(q * q, axis=-1)
    np.testing.assert_allclose(np.sum(qh * qh, axis=-1), s / (s + prep.EPS), rtol=1e-13)
    # direction preserved
    cos = np.sum(qh * q, axis=-1) / np.sqrt(np.sum(qh * qh, axis=-1) * s)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-13)
    # scale invariance when eps is negligible
    np.testing.assert_allclose(prep.normalize(7.5 * q, eps=0.0), prep.normalize(q, eps=0.0),
                               rtol=1e-13)
    z = np.zeros((2, 16))
    assert np.array_equal(prep.normalize(z), z)


def raw_inputs(variant, B=2, T=9, H=2, dk=3, dv=2, seed=11):
    r = np.random.default_rng(seed)
    x = dict(q=r.standard_normal((B, T, H, dk)) * 2.0,
             k=r.standard_normal((B, T, H, dk)) * 0.7,
             v=r.standard_normal((B, T, H, dv)),
             b=r.standard_normal((B, T, H)),
             x=None,
             h0=0.3 * r.standard_normal((B, H, dk, dv)),
             dO=r.standard_normal((B, T, H, dv)),
             dhT=r.standard_normal((B, H, dk, dv)))
    if variant == "gdn":
        x["x"] = r.standard_normal((B, T, H)) - 1.0
    elif variant == "kda":
        x["x"] = r.standard_normal((B, T, H, dk)) - 1.0
    return x


def raw_loss(variant, x, scale):
    o, hT = prep.forward_raw(variant, x["q"], x["k"], x["v"], x["b"], x["x"], x["h0"],
                             scale=scale)
    return float(np.sum(o * x["dO"]) + np.sum(hT * x["dhT"]))


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
def test_raw_gradients_match_central_differences(variant):
    scale = 0.8
    x = raw_inputs(variant)
    grads = prep.backward_raw(variant, x["q"], x["k"], x["v"], x["b"], x["x"], x["h0"],
                              x["dO"], x["dhT"], scale=scale)
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("b", "dbeta"), ("h0", "dh0")]
    if variant != "deltanet":
        names.append(("x", "dg"))
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
            lp = raw_loss(variant, xp, scale)
            xp[name][idx] -= 2 * h
            lm = raw_loss(variant, xp, scale)
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(grads[gname] - fd)) / max(1.0, np.max(np.abs(fd)))
        assert err < 1e-6, f"{variant} {gname}: relative error {err}"


def test_raw_forward_equals_prepared_forward():
    # the composite is the recurrence on the mapped tensors, nothing more
    x = raw_inputs("kda")
    o1, h1 = prep.forward_raw("kda", x["q"], x["k"], x["v"], x["b"], x["x"], x["h0"])
    q = x["q"] / np.linalg.norm(x["q"], axis=-1, keepdims=True)
    k = x["k"] / np.linalg.norm(x["k"], axis=-1, keepdims=True)
    beta = np.exp(x["b"]) / (1.0 + np.exp(x["b"]))
    g = np.log(1.0 / (1.0 + np.exp(x["x"])))
    o2, h2 = oracle.forward("kda", q, k, x["v"], beta, g, x["h0"])
    # eps = 1e-6 against |q|^2 of order 10 moves the result by < 1e-6 relative
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-5)
    np.testing.assert_allclose(h1, h2, rtol=0, atol=1e-5)
