"""Helpers shared by the GPU parity tests: run the library through the C ABI
and the fp64 oracle on the same seeded inputs, and compare element by element.

Tolerance (written here, used by every parity test):
  * fp32 inputs: max |gpu - oracle| <= 1e-4 on every output and gradient.
  * bf16 inputs (fp32 accumulation, fp32-written outputs), per tensor:
        max |gpu - oracle| <= max(2e-2, 1e-2 * max |oracle|)
    i.e. the stated 2e-2 absolute for every tensor whose entries stay within +-2
    (o, hT, dh0 and dv of every workload here), and 1e-2 of the tensor's
    largest entry beyond that.  The bf16 path rounds every intermediate operand
    of its tensor-core products (decayed keys and queries, the UT inverse, the
    WY factors, the state, the writes and their gradients) to bf16, a relative
    2^-9 each; the gradients dq, dk, dbeta, dg reach 10-90 at T = 4096 and
    their measured full-size error is 3-7e-3 of the tensor's largest entry
    (0.06-0.08 absolute for Gated DeltaNet and KDA, up to 0.46 for DeltaNet,
    whose gradients grow largest).  The relative term is about 1.5x that
    measured error: loose enough for rounding, tight enough that a dropped
    term or a wrong index (errors of the size of the values) fails.
Every comparison is recorded (absolute error, largest reference entry, bound)
and summarised at the end of the run.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from delta_rule_recurrent_gated_gb300 import binding, inputs

FIELDS = ("o", "hT", "dq", "dk", "dv", "dbeta", "dg", "dh0")

F32_ABS = 1e-4
BF16_ABS = 2e-2
BF16_REL = 1e-2

# (test, workload, tensor, max abs error, max |reference|, bound) of every comparison
RECORDS: list = []


def record(w, name: str, err: float, ref_max: float, tol: float):
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    RECORDS.append((test, w.name, w.io, name, float(err), float(ref_max), float(tol)))


def summary_lines():
    """Worst absolute error per (workload, tensor) over the recorded comparisons."""
    worst = {}
    for test, wname, io, name, err, rmax, tol in RECORDS:
        key = (wname, io)
        d = worst.setdefault(key, {})
        if name not in d or err / tol > d[name][0] / d[name][2]:
            d[name] = (err, rmax, tol)
    out = []
    for (wname, io), d in sorted(worst.items()):
        parts = [f"{n} {e:.1e}/{t:.1e} (|ref| {r:.2g})" for n, (e, r, t) in d.items()]
        out.append(f"{wname} [{io}]: " + "; ".join(parts))
    log = os.environ.get("DR_PARITY_LOG")
    if log:
        with open(log, "w") as f:
            for r in RECORDS:
                f.write(json.dumps(dict(zip(("test", "workload", "io", "tensor", "max_abs_err",
                                             "max_abs_ref", "bound"), r))) + "\n")
    return out


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
        return F32_ABS
    return max(BF16_ABS, BF16_REL * (float(np.max(np.abs(ref))) if ref.size else 0.0))


def check(w, name: str, got: np.ndarray, ref: np.ndarray):
    """Max-abs error of one tensor against its bound, recorded; returns (err, tol)."""
    assert np.all(np.isfinite(got)), f"{w.name} {name}: non-finite values"
    err = float(np.max(np.abs(got.astype(np.float64) - ref))) if ref.size else 0.0
    tol = tolerance(w, ref)
    record(w, name, err, float(np.max(np.abs(ref))) if ref.size else 0.0, tol)
    return err, tol


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
        err, tol = check(w, n, g, r)
        report[n] = (err, tol, err / max(float(np.max(np.abs(r))) if r.size else 0.0, 1e-30))
    bad = {n: v for n, v in report.items() if not v[0] <= v[1]}
    assert not bad, f"{w.name}: over tolerance (abs err, bound, rel err): {bad}; all: {report}"
    return report
