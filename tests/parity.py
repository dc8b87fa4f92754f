"""Helpers shared by the GPU parity tests: run the library through the C ABI
and the fp64 oracle on the same seeded inputs, and compare element by element.

Tolerance (written here, used by every parity test):
  * fp32 inputs: max |gpu - oracle| <= 1e-4 on every output and gradient.
  * bf16 inputs (fp32 accumulation, fp32-written outputs):
        max |gpu - oracle| <= 2e-2 * max(1, max |oracle|)   per tensor,
    i.e. 2e-2 absolute for tensors whose entries stay within +-1 and 2e-2
    relative to the tensor's largest entry beyond that.  bf16 operands carry
    a relative rounding of 2^-9 into every tensor-core product, so the error of
    a large-magnitude gradient scales with its magnitude; the absolute error is
    reported alongside in the failure message.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from delta_rule_recurrent_gated_gb300 import binding, inputs

FIELDS = ("o", "hT", "dq", "dk", "dv", "dbeta", "dg", "dh0")


def to_dev(x, dev):
    return {n: (val.to(dev) if torch.is_tensor(val) and n != "cu_seqlens" else val)
            for n, val in x.items()}


def run_gpu(w: inputs.Workload, x: dict, reuse=True, out="f32", grad="f32", dev="cuda",
            prob=None, backward=True):
    if prob is None:
        prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io,
                               out=out, grad=grad, scale=w.scale, cu_seqlens=x["cu_seqlens"],
                               device=dev)
    t = to_dev(x, dev)
    o, hT = prob.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
    res = {"o": o, "hT": hT}
    if backward:
        gr = prob.backward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], t["dO"],
                           t["dhT"], reuse_fwd=reuse)
        res.update(gr)
    torch.cuda.synchronize()
    st = prob.status()
    assert st == binding.DR_OK, binding.error_string(st)
    # fp32 on the host is exact for the fp32 / bf16 values the library writes
    return {n: (None if val is None else val.float().cpu().numpy()) for n, val in res.items()}


def run_oracle(w: inputs.Workload, x: dict, units=None, backward=True):
    a = dict(q=x["q"], k=x["k"], v=x["v"], beta=x["beta"], g=x["g"], h0=x["h0"],
             scale=w.scale, cu_seqlens=x["cu_seqlens"], units=units)
    o, hT = oracle.forward(w.variant, **a)
    res = {"o": o, "hT": hT}
    if backward:
        res.update(oracle.backward(w.variant, dO=x["dO"], dhT=x["dhT"], **a))
    return res


def tolerance(w: inputs.Workload, ref: np.ndarray) -> float:
    if w.io == "f32":
        return 1e-4
    return 2e-2 * max(1.0, float(np.max(np.abs(ref))) if ref.size else 1.0)


def unit_mask(w, x, units, name, shape):
    """Boolean mask selecting the entries of `name` that belong to `units`."""
    H = w.H
    m = np.zeros(shape, dtype=bool)
    cu = x["cu_seqlens"]
    for u in units:
        n, h = divmod(int(u), H)
        if name in ("hT", "dh0"):
            m[n, h] = True
        else:
            if cu is None:
                m[n, :, h] = True
            else:
                lo, hi = int(cu[n]), int(cu[n + 1])
                m[0, lo:hi, h] = True
    return m


def compare(w, x, got: dict, ref: dict, units=None, fields=FIELDS):
    report = {}
    for n in fields:
        if ref.get(n) is None or got.get(n) is None:
            continue
        r, g = ref[n], got[n]
        assert r.shape == g.shape, (n, r.shape, g.shape)
        if units is not None:
            m = unit_mask(w, x, units, n, r.shape)
            r, g = r[m], g[m]
        assert np.all(np.isfinite(g)), f"{n}: non-finite values"
        err = float(np.max(np.abs(g.astype(np.float64) - r))) if r.size else 0.0
        tol = tolerance(w, r)
        report[n] = (err, tol)
    bad = {n: v for n, v in report.items() if not v[0] <= v[1]}
    assert not bad, f"{w.name}: over tolerance (err, tol): {bad}; all: {report}"
    return report
