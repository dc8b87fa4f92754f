"""Why the bf16 path's bound is relative for the large gradients (CPU only).

tests/bf16_emulation.py restates the chunkwise algebra of the bf16 kernels in fp64
and rounds to bf16 exactly the intermediates the kernels keep as bf16 operands.
Pinned first: without rounding it reproduces the fp64 oracle.  Then, on one full
(sequence, head) unit of the Gated DeltaNet layer shape (T = 4096, d = 128, h0):
  * with the kernels' bf16 rounding, o and hT meet 2e-2 absolute, while dq, dk,
    dbeta and dg (entries up to ~15) miss it, at well under 1e-2 of their largest
    entry: the error the parity bound of tests/parity.py is built around;
  * holding only the state-side operands (S, dS, U, dU, T and their images) in
    two-term bf16 splits leaves those gradient errors above 2e-2: the error is
    spread over the chunk-local intermediates as well;
  * holding every intermediate in a two-term split (about 16 mantissa bits) meets
    2e-2 absolute on every tensor: what the absolute bound would need.
"""
import numpy as np
import pytest

import oracle
from delta_rule_recurrent_gated_gb300 import inputs

import bf16_emulation as emu

GRADS = ("dq", "dk", "dbeta", "dg")


def unit(w, seed):
    x = inputs.make(w, seed=seed)
    f = lambda t: None if t is None else t[0, :, 0].double().numpy()
    st = lambda t: None if t is None else t[0, 0].double().numpy()
    u = dict(q=f(x["q"]), k=f(x["k"]), v=f(x["v"]), beta=f(x["beta"]), g=f(x["g"]),
             h0=st(x["h0"]), dO=f(x["dO"]), dhT=st(x["dhT"]))
    a = dict(q=x["q"][:1], k=x["k"][:1], v=x["v"][:1], beta=x["beta"][:1],
             g=None if x["g"] is None else x["g"][:1], h0=None if x["h0"] is None else x["h0"][:1],
             scale=w.scale, units=np.array([0], dtype=np.int32))
    o, hT = oracle.forward(w.variant, **a)
    gr = oracle.backward(w.variant, dO=x["dO"][:1],
                         dhT=None if x["dhT"] is None else x["dhT"][:1], **a)
    ref = dict(o=o[0, :, 0], hT=hT[0, 0])
    for n, val in gr.items():
        ref[n] = None if val is None else (val[0, 0] if n == "dh0" else val[0, :, 0])
    return u, ref


def errors(w, u, ref, rnd):
    o, hT, gr = emu.run_unit(rnd, w.variant, u["q"], u["k"], u["v"], u["beta"], u["g"],
                             u["h0"], u["dO"], u["dhT"], w.scale, w.chunk)
    got = dict(o=o, hT=hT, **gr)
    return {n: (float(np.max(np.abs(got[n] - r))), float(np.max(np.abs(r))))
            for n, r in ref.items() if r is not None}


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
def test_emulation_without_rounding_is_the_oracle(variant):
    w = inputs.small(variant, B=1, T=200, H=1, dk=32, dv=32)
    u, ref = unit(w, seed=81)
    for n, (err, mx) in errors(w, u, ref, emu.Rounding()).items():
        assert err <= 1e-11 * max(1.0, mx), (n, err)


@pytest.fixture(scope="module")
def headline_unit():
    w = inputs.replace(inputs.get("gdn_h0_b8_t4096_h16_d128"), B=1, H=1)
    u, ref = unit(w, seed=0)
    return w, u, ref


def test_kernel_rounding_misses_the_absolute_bound_on_the_gradients(headline_unit):
    w, u, ref = headline_unit
    e = errors(w, u, ref, emu.Rounding(bf=emu.ALL_POINTS))
    assert e["o"][0] <= 2e-2 and e["hT"][0] <= 2e-2
    assert max(e[n][0] for n in GRADS) > 2e-2
    for n in GRADS:
        assert e[n][0] <= 1e-2 * e[n][1], (n, e[n])


def test_state_side_split_alone_does_not_reach_it(headline_unit):
    w, u, ref = headline_unit
    e = errors(w, u, ref, emu.Rounding(bf=emu.ALL_POINTS, split=emu.STATE_POINTS))
    assert max(e[n][0] for n in GRADS) > 2e-2


def test_every_intermediate_split_reaches_it(headline_unit):
    w, u, ref = headline_unit
    e = errors(w, u, ref, emu.Rounding(split=emu.ALL_POINTS))
    for n, (err, _) in e.items():
        assert err <= 2e-2, (n, err)
