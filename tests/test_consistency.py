"""GPU consistency of the state interface and of unit independence, through the C ABI.

* Checkpoint / resume: a sequence run as two calls, the first call's final state
  passed as the second call's initial state (and, backward, the second call's dh0
  passed as the first call's dhT), gives the outputs and gradients of one call, at a
  split on a chunk boundary and at one inside a chunk.
* Independence: a NaN placed in one (sequence, head) stays in that unit; every other
  unit matches the oracle.
Tolerance: tests/parity.py."""
import numpy as np
import pytest
import torch

from delta_rule_recurrent_gated_gb300 import binding, inputs

from parity import compare, run_oracle, tolerance

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dbeta", "dg")


def _call(w, x, T, h0, dhT):
    """One forward + backward of the first T tokens of x with the given h0 / dhT."""
    prob = binding.Problem(w.variant, w.B, T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io,
                           device="cuda")
    t = {n: (v.cuda() if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    o, hT = prob.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], h0)
    gr = prob.backward(t["q"], t["k"], t["v"], t["beta"], t["g"], h0, t["dO"], dhT,
                       reuse_fwd=True)
    torch.cuda.synchronize()
    assert prob.status() == binding.DR_OK
    return o, hT, gr


def _cut(x, lo, hi):
    out = dict(x)
    for n in ("q", "k", "v", "beta", "g", "dO"):
        if x[n] is not None:
            out[n] = x[n][:, lo:hi].contiguous()
    return out


@pytest.mark.parametrize("variant", ["gdn", "kda"])
@pytest.mark.parametrize("split", [128, 100])
def test_two_calls_through_the_state_equal_one(variant, split):
    w = inputs.small(variant, B=2, T=230, H=2, dk=128, dv=128)
    x = inputs.make(w, seed=61)
    h0 = x["h0"].cuda()
    dhT = x["dhT"].cuda()
    # one call
    o1, hT1, g1 = _call(w, x, w.T, h0, dhT)
    # two calls: [0, split) then [split, T)
    a, b = _cut(x, 0, split), _cut(x, split, w.T)
    _, hTa, _ = _call(inputs.replace(w, T=split), a, split, h0, None)  # forward state only
    ob, hTb, gb = _call(inputs.replace(w, T=w.T - split), b, w.T - split, hTa, dhT)
    oa, _, ga = _call(inputs.replace(w, T=split), a, split, h0, gb["dh0"])
    ref = run_oracle(w, x)
    got = {"o": torch.cat([oa, ob], 1), "hT": hTb, "dh0": ga["dh0"]}
    for n in GRADS:
        got[n] = torch.cat([ga[n], gb[n]], 1)
    got = {n: v.float().cpu().numpy() for n, v in got.items()}
    compare(w, x, got, ref)
    # and against the single call itself
    one = {"o": o1, "hT": hT1, **g1}
    for n in ("o", "hT", "dh0") + GRADS:
        d = float((one[n].float().cpu() - torch.from_numpy(got[n])).abs().max())
        assert d <= tolerance(w, ref[n]), (n, d)


@pytest.mark.parametrize("variant", ["deltanet", "kda"])
def test_nan_stays_in_its_unit(variant):
    w = inputs.small(variant, B=2, T=150, H=3, dk=64, dv=64)
    x = inputs.make(w, seed=62)
    x["v"] = x["v"].clone()
    x["v"][1, 70, 2, 5] = float("nan")  # sequence 1, head 2
    prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, device="cuda")
    t = {n: (v.cuda() if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    o, hT = prob.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
    gr = prob.backward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], t["dO"], t["dhT"],
                       reuse_fwd=True)
    torch.cuda.synchronize()
    assert prob.status() == binding.DR_OK
    got = {"o": o, "hT": hT, **gr}
    got = {n: (None if v is None else v.float().cpu().numpy()) for n, v in got.items()}
    clean = [n * w.H + h for n in range(w.B) for h in range(w.H) if (n, h) != (1, 2)]
    ref = run_oracle(w, x, units=np.array(clean, dtype=np.int32))
    compare(w, x, got, ref, units=clean)
    assert not np.all(np.isfinite(got["o"][1, :, 2]))  # the poisoned unit shows it
