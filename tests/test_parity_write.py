"""GPU parity of the emitted write u = beta r (dr_fwd_u) and of the gradients
with its incoming gradient dU (dr_bwd_u) against the fp64 oracle, through the C
ABI: tensor-core path (bf16) with the backward reusing or recomputing the
forward's residuals, and the fp32 path; ragged tails and packed sequences.
Tolerance: tests/parity.py."""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_recurrent_gated_gb300 import binding, inputs

from parity import check

pytestmark = pytest.mark.gpu

VARIANTS = ["deltanet", "gdn", "kda"]


def _run(w, x, dU_host, reuse=True):
    dev = torch.device("cuda:0")
    t = {n: (v.to(dev) if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io,
                           out="f32", grad="f32", scale=w.scale, cu_seqlens=x["cu_seqlens"],
                           device=dev)
    u = torch.empty(w.B, w.T, w.H, w.dv, dtype=torch.float32, device=dev)
    o, hT = prob.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], u=u)
    gr = prob.backward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], t["dO"], t["dhT"],
                       reuse_fwd=reuse, dU=dU_host.to(dev))
    torch.cuda.synchronize()
    assert prob.status() == binding.DR_OK
    res = {"o": o, "hT": hT, "u": u, **gr}
    return {n: (None if v is None else v.float().cpu().numpy()) for n, v in res.items()}


def _oracle(w, x, dU):
    a = dict(q=x["q"], k=x["k"], v=x["v"], beta=x["beta"], g=x["g"], h0=x["h0"],
             scale=w.scale, cu_seqlens=x["cu_seqlens"])
    o, hT, u = oracle.forward(w.variant, want_u=True, **a)
    res = {"o": o, "hT": hT, "u": u}
    res.update(oracle.backward(w.variant, dO=x["dO"], dhT=x["dhT"], dU=dU, **a))
    return res


def _compare(w, got, ref):
    for name, r in ref.items():
        if r is None:
            continue
        err, tol = check(w, name, got[name], r)
        assert err <= tol, f"{w.name} {name}: err {err} > tol {tol}"


def _dU(w, x, seed):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if w.io == "bf16" else torch.float32
    return torch.randn(x["v"].shape, generator=g).to(dt)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("io,d,chunk", [("bf16", 128, 64), ("bf16", 64, 64), ("f32", 32, 16)])
@pytest.mark.parametrize("reuse", [True, False])
def test_write_and_its_gradient(variant, io, d, chunk, reuse):
    w = inputs.small(variant, B=2, T=150, H=2, dk=d, dv=d, chunk=chunk, io=io)
    x = inputs.make(w, seed=31)
    dU = _dU(w, x, 32)
    _compare(w, _run(w, x, dU, reuse), _oracle(w, x, dU.double().numpy()))


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_write_packed_sequences(variant):
    w = inputs.small(variant, H=2, dk=128, dv=128, lengths=[100, 0, 64, 1, 191, 7])
    x = inputs.make(w, seed=33)
    dU = _dU(w, x, 34)
    _compare(w, _run(w, x, dU), _oracle(w, x, dU.double().numpy()))


def test_write_gradient_alone():
    """dO = 0 and no dhT: every gradient comes from dU through the write."""
    w = inputs.small("kda", B=2, T=130, H=2, dk=128, dv=128, dhT=False)
    x = inputs.make(w, seed=35)
    x["dO"] = torch.zeros_like(x["dO"])
    dU = _dU(w, x, 36)
    _compare(w, _run(w, x, dU), _oracle(w, x, dU.double().numpy()))
