"""GPU parity of the recurrent step (dr_decode) against the fp64 oracle, through
the C ABI.  The oracle's forward is the token-by-token recurrence itself, so a
run of single-token calls that carry the state must reproduce its outputs for
every token and its final state; one multi-token call must do the same.
Tolerance: tests/parity.py (fp32 inputs 1e-4; bf16 inputs 2e-2 relative to the
tensor's magnitude beyond 1; outputs written in fp32)."""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_recurrent_gated_gb300 import binding, inputs

from parity import check

pytestmark = pytest.mark.gpu

VARIANTS = ["deltanet", "gdn", "kda"]


def _oracle(w, x):
    return oracle.forward(w.variant, q=x["q"], k=x["k"], v=x["v"], beta=x["beta"], g=x["g"],
                          h0=x["h0"], scale=w.scale)


def _check(w, name, got, ref):
    err, tol = check(w, name, got, ref)
    assert err <= tol, f"{w.name} {name}: err {err} > tol {tol}"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("io,d", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 32),
                                  ("f32", 16)])
def test_single_token_steps_match_the_recurrence(variant, io, d):
    w = inputs.replace(inputs.small(variant, B=3, T=7, H=2, dk=d, dv=d, io=io), scale=0.5)
    x = inputs.make(w, seed=21, need_grad_inputs=False)
    o_ref, h_ref = _oracle(w, x)
    dev = torch.device("cuda:0")
    dec = binding.Decoder(variant, w.B, 1, w.H, d, d, io=io, out="f32", scale=w.scale, device=dev)
    state = x["h0"].to(dev).clone()
    outs = []
    for t in range(w.T):
        sl = slice(t, t + 1)
        q, k, v = (x[n][:, sl].contiguous().to(dev) for n in ("q", "k", "v"))
        beta = x["beta"][:, sl].contiguous().to(dev)
        g = None if x["g"] is None else x["g"][:, sl].contiguous().to(dev)
        outs.append(dec.step(q, k, v, beta, g, state))
    torch.cuda.synchronize()
    o = torch.cat(outs, dim=1).cpu().numpy()
    _check(w, "o", o, o_ref)
    _check(w, "state", state.cpu().numpy(), h_ref)


@pytest.mark.parametrize("variant", VARIANTS)
def test_multi_token_call_and_zero_tokens(variant):
    w = inputs.small(variant, B=2, T=33, H=3, dk=64, dv=64, io="bf16")
    x = inputs.make(w, seed=22, need_grad_inputs=False)
    o_ref, h_ref = _oracle(w, x)
    dev = torch.device("cuda:0")
    t = {n: (v.to(dev) if torch.is_tensor(v) else v) for n, v in x.items()}
    state = t["h0"].clone()
    dec = binding.Decoder(variant, w.B, w.T, w.H, 64, 64, io="bf16", out="f32", device=dev)
    o = dec.step(t["q"], t["k"], t["v"], t["beta"], t["g"], state)
    torch.cuda.synchronize()
    _check(w, "o", o.cpu().numpy(), o_ref)
    _check(w, "state", state.cpu().numpy(), h_ref)
    # T = 0 leaves the state untouched
    before = state.clone()
    empty = binding.Decoder(variant, w.B, 0, w.H, 64, 64, io="bf16", out="f32", device=dev)
    e = lambda n: t[n][:, :0].contiguous() if t[n] is not None else None
    empty.step(e("q"), e("k"), e("v"), e("beta"), e("g"), state)
    torch.cuda.synchronize()
    assert torch.equal(state, before)


def test_decode_at_serving_batch_sampled():
    """B = 256 sequences x 16 heads at d = 128 (a 256 MiB state), one bf16 token per
    call: sampled (sequence, head) units against the oracle."""
    w = inputs.small("kda", B=256, T=1, H=16, dk=128, dv=128, io="bf16")
    x = inputs.make(w, seed=23, need_grad_inputs=False)
    dev = torch.device("cuda:0")
    t = {n: (v.to(dev) if torch.is_tensor(v) else v) for n, v in x.items()}
    state = t["h0"].clone()
    dec = binding.Decoder("kda", w.B, 1, w.H, 128, 128, io="bf16", out="f32", device=dev)
    o = dec.step(t["q"], t["k"], t["v"], t["beta"], t["g"], state).cpu().numpy()
    torch.cuda.synchronize()
    s = state.cpu().numpy()
    rng = np.random.default_rng(0)
    for n in sorted(rng.choice(w.B, size=4, replace=False)):
        a = {m: (None if x[m] is None else x[m][n:n + 1]) for m in ("q", "k", "v", "beta", "g", "h0")}
        o_ref, h_ref = oracle.forward("kda", scale=w.scale, **a)
        _check(w, f"o[{n}]", o[n:n + 1], o_ref)
        _check(w, f"state[{n}]", s[n:n + 1], h_ref)
