"""fp64 oracle of the input preparation in front of the delta-rule memory.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use it.

The pages give the recurrence on prepared inputs: q and k are unit-norm keys,
beta a write strength in [0, 1] and alpha = e^g a decay in (0, 1] ("Linear
Attention Architectures: Mechanisms, Trade-offs, and Cross-Layer Routing",
section "Metodologia y Marco de Trabajo", item 1, the DeltaNet / Gated DeltaNet /
Kimi Delta Attention bullets).  The maps that produce them from a layer's
projections are the standard ones of these layers, as the workloads draw them:

  q_hat = q / sqrt(sum_c q_c^2 + eps)      per (token, head), eps = 1e-6 (reading:
                                           eps guards the zero vector)
  k_hat = k / sqrt(sum_c k_c^2 + eps)
  beta  = sigmoid(b) = 1 / (1 + e^-b)
  g     = log alpha = -softplus(x) = -log(1 + e^x)

``chain`` maps the gradients of a loss with respect to (q_hat, k_hat, beta, g)
to gradients with respect to the raw (q, k, b, x) by the derivative of each map,
written out by hand:

  d q = (d q_hat - q_hat (q_hat . d q_hat)) / sqrt(|q|^2 + eps)
  d b = d beta * beta (1 - beta)
  d x = -d g * sigmoid(x)

Parity status: pinned by ``tests/test_oracle_prepare.py`` (closed-form values of
the three maps, the unit norm and the scale invariance of the normalisation, and
central finite differences of the composite loss with respect to the raw
inputs, which check ``chain`` without using its formulas).
"""
from __future__ import annotations

import numpy as np

from . import backward as _backward
from . import forward as _forward
from . import _f64

EPS = 1e-6


def normalize(x, eps=EPS):
    """x / sqrt(sum over the last axis of x^2 + eps), fp64."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def sigmoid(b):
    b = _f64(b)
    return 1.0 / (1.0 + np.exp(-b))


def neg_softplus(x):
    """-log(1 + e^x), written as -(max(x, 0) + log1p(e^-|x|)) so that it does not
    overflow for large x."""
    x = _f64(x)
    return -(np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x))))


def prepare(variant, q, k, b, x, eps=EPS):
    """(q_hat, k_hat, beta, g) from the raw tensors; g is None for DeltaNet."""
    g = None if x is None or variant in ("deltanet", 0) else neg_softplus(x)
    return normalize(q, eps), normalize(k, eps), sigmoid(b), g


def _chain_norm(x, dn, eps):
    x = _f64(x)
    rinv = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    xh = x * rinv
    return rinv * (dn - xh * np.sum(xh * dn, axis=-1, keepdims=True))


def chain(variant, q, k, b, x, grads, eps=EPS):
    """Gradients with respect to the raw (q, k, b, x), from ``grads`` (a dict with
    dq, dk, dbeta, dg with respect to the prepared tensors; other keys copied)."""
    out = dict(grads)
    out["dq"] = _chain_norm(q, grads["dq"], eps)
    out["dk"] = _chain_norm(k, grads["dk"], eps)
    s = sigmoid(b)
    out["dbeta"] = grads["dbeta"] * s * (1.0 - s)
    if grads.get("dg") is not None:
        out["dg"] = -grads["dg"] * sigmoid(x)
    return out


def forward_raw(variant, q, k, v, b, x=None, h0=None, eps=EPS, **kw):
    """The oracle forward on prepared inputs; same returns as ``oracle.forward``."""
    qh, kh, beta, g = prepare(variant, q, k, b, x, eps)
    return _forward(variant, qh, kh, v, beta, g, h0, **kw)


def backward_raw(variant, q, k, v, b, x, h0, dO, dhT=None, eps=EPS, **kw):
    """Gradients of the same loss as ``oracle.backward`` with respect to the raw
    q, k, b, x (and v, h0 unchanged)."""
    qh, kh, beta, g = prepare(variant, q, k, b, x, eps)
    grads = _backward(variant, qh, kh, v, beta, g, h0, dO, dhT, **kw)
    return chain(variant, q, k, b, x, grads, eps)
