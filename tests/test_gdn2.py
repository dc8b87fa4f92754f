"""GPU parity of Gated DeltaNet-2 (dr_gdn2_fwd / dr_gdn2_bwd, the fp32 CUDA-core
chunkwise path) against the fp64 oracle (oracle/dro2.c), through the C ABI: o, hT
and every gradient (dq, dk, dv, derase, dwrite, dg, dh0) element by element.
Covers fp32 and bf16 inputs, every supported d and chunk, ragged tails, packed
sequences with an empty one, a zero-token call, the reduction to Gated DeltaNet
(erase = write = beta gives the library's own Gated DeltaNet results), and the full
workload size on sampled (sequence, head) units.  Tolerance: tests/parity.py.
The variant's equations are a reading of the pages (oracle/dro2.c states it)."""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_recurrent_gated_gb300 import binding, inputs

from parity import check, tolerance

pytestmark = pytest.mark.gpu

FIELDS = ("o", "hT", "dq", "dk", "dv", "derase", "dwrite", "dg", "dh0")


def run_gpu(w, x, out="f32", grad="f32", reuse=True):
    prob = binding.Gdn2Problem(w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io, out=out,
                               grad=grad, scale=w.scale, cu_seqlens=x["cu_seqlens"])
    t = {n: (v.cuda() if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    o, hT = prob.forward(t["q"], t["k"], t["v"], t["erase"], t["write"], t["g"], t["h0"])
    gr = prob.backward(t["q"], t["k"], t["v"], t["erase"], t["write"], t["g"], t["h0"], t["dO"],
                       t["dhT"], reuse_fwd=reuse)
    torch.cuda.synchronize()
    assert prob.status() == binding.DR_OK
    res = {"o": o, "hT": hT, **gr}
    return {n: v.float().cpu().numpy() for n, v in res.items()}


def run_oracle(w, x, units=None):
    a = dict(scale=w.scale, cu_seqlens=x["cu_seqlens"], units=units)
    o, hT = oracle.forward_gdn2(x["q"], x["k"], x["v"], x["erase"], x["write"], x["g"], x["h0"],
                                **a)
    res = {"o": o, "hT": hT}
    res.update(oracle.backward_gdn2(x["q"], x["k"], x["v"], x["erase"], x["write"], x["g"],
                                    x["h0"], x["dO"], x["dhT"], **a))
    return res


def compare(w, got, ref):
    bad = {}
    for n in FIELDS:
        r, g = ref[n], got[n]
        assert r.shape == g.shape, (n, r.shape, g.shape)
        err, tol = check(w, n, g, r)
        if not err <= tol:
            bad[n] = (err, tol)
    assert not bad, f"{w.name}: over tolerance {bad}"


@pytest.mark.parametrize("io,d,chunk", [("f32", 16, 16), ("f32", 32, 32), ("f32", 64, 64),
                                        ("f32", 64, 16), ("bf16", 64, 64), ("bf16", 32, 64)])
def test_fwd_bwd_small(io, d, chunk):
    w = inputs.replace(inputs.small("gdn2", B=2, T=150, H=2, dk=d, dv=d, chunk=chunk, io=io),
                       scale=0.8)
    x = inputs.make_gdn2(w, seed=41)
    compare(w, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("T", [1, 63, 64, 65])
def test_short_and_tail(T):
    w = inputs.small("gdn2", B=2, T=T, H=2, dk=32, dv=16, chunk=64, io="f32", h0=False,
                     dhT=False)
    x = inputs.make_gdn2(w, seed=42)
    compare(w, run_gpu(w, x), run_oracle(w, x))


def test_packed():
    w = inputs.small("gdn2", H=2, dk=64, dv=64, chunk=64, io="f32",
                     lengths=[100, 0, 64, 1, 131, 7])
    x = inputs.make_gdn2(w, seed=43)
    compare(w, run_gpu(w, x), run_oracle(w, x))


def test_reduces_to_gated_deltanet_on_the_gpu():
    """erase = write = beta: the Gated DeltaNet-2 kernels give the library's own Gated
    DeltaNet results (fp32 path), and dbeta = sum of the gate gradients."""
    w = inputs.small("gdn", B=2, T=130, H=2, dk=32, dv=32, chunk=32, io="f32")
    x = inputs.make(w, seed=44)
    pg = binding.Problem("gdn", w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io="f32")
    t = {n: (v.cuda() if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    o1, h1 = pg.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
    g1 = pg.backward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], t["dO"], t["dhT"])
    erase = t["beta"][..., None].expand(*t["beta"].shape, w.dk).contiguous()
    write = t["beta"][..., None].expand(*t["beta"].shape, w.dv).contiguous()
    p2 = binding.Gdn2Problem(w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io="f32")
    o2, h2 = p2.forward(t["q"], t["k"], t["v"], erase, write, t["g"], t["h0"])
    g2 = p2.backward(t["q"], t["k"], t["v"], erase, write, t["g"], t["h0"], t["dO"], t["dhT"])
    torch.cuda.synchronize()
    for a, b, n in ((o1, o2, "o"), (h1, h2, "hT")):
        assert float((a - b).abs().max()) <= 1e-4, n
    for n in ("dq", "dk", "dv", "dg", "dh0"):
        assert float((g1[n] - g2[n]).abs().max()) <= 1e-4, n
    dbeta = g2["derase"].sum(-1) + g2["dwrite"].sum(-1)
    assert float((dbeta - g1["dbeta"]).abs().max()) <= 1e-4


def test_zero_tokens_pass_the_state_through():
    w = inputs.small("gdn2", B=2, T=0, H=2, dk=16, dv=16, chunk=16, io="f32")
    x = inputs.make_gdn2(w, seed=45)
    got = run_gpu(w, x)
    np.testing.assert_array_equal(got["hT"], x["h0"].numpy())
    np.testing.assert_array_equal(got["dh0"], x["dhT"].numpy())


def test_full_size_sampled():
    w = inputs.get("gdn2_b4_t2048_h8_d64")
    x = inputs.make_gdn2(w, seed=0)
    got = run_gpu(w, x)
    rng = np.random.default_rng(2)
    units = sorted(int(u) for u in rng.choice(w.B * w.H, size=3, replace=False))
    ref = run_oracle(w, x, units=np.array(units, dtype=np.int32))
    for u in units:
        n, h = divmod(u, w.H)
        for name in FIELDS:
            r = ref[name][n, h] if name in ("hT", "dh0") else ref[name][n, :, h]
            g = got[name][n, h] if name in ("hT", "dh0") else got[name][n, :, h]
            err, tol = check(w, name, g, r)
            assert err <= tol, f"unit {u} {name}: err {err}"


@pytest.mark.parametrize("io,d", [("bf16", 128), ("f32", 64), ("f32", 16)])
def test_decode_steps_match_the_recurrence(io, d):
    """dr_gdn2_decode token by token (state carried between calls) and as one
    multi-token call reproduce the oracle's outputs and final state."""
    w = inputs.replace(inputs.small("gdn2", B=3, T=9, H=2, dk=d, dv=d, io=io), scale=0.5)
    x = inputs.make_gdn2(w, seed=46, need_grad_inputs=False)
    o_ref, h_ref = oracle.forward_gdn2(x["q"], x["k"], x["v"], x["erase"], x["write"], x["g"],
                                       x["h0"], scale=w.scale)
    dev = torch.device("cuda:0")
    for per_token in (True, False):
        T = 1 if per_token else w.T
        dec = binding.Decoder("gdn2", w.B, T, w.H, d, d, io=io, out="f32", scale=w.scale,
                              device=dev)
        state = x["h0"].to(dev).clone()
        outs = []
        for t0 in range(0, w.T, T):
            sl = slice(t0, t0 + T)
            args = [x[n][:, sl].contiguous().to(dev) for n in ("q", "k", "v", "erase", "write", "g")]
            outs.append(dec.step_gdn2(*args, state))
        torch.cuda.synchronize()
        o = torch.cat(outs, dim=1).cpu().numpy()
        for name, got, ref in (("o", o, o_ref), ("state", state.cpu().numpy(), h_ref)):
            err, tol = check(w, name, got, ref)
            assert err <= tol, f"{name} per_token={per_token}: err {err}"


def test_bf16_gradients_and_rerun_bit_identical():
    """bf16-written outputs and gradients stay within the bf16 reading of the tolerance
    (half an ulp of bf16 on top of 2e-2); two runs are bit-identical (the slices' partial
    gradients are added in a fixed order)."""
    w = inputs.small("gdn2", B=2, T=130, H=2, dk=64, dv=64, chunk=64, io="bf16")
    x = inputs.make_gdn2(w, seed=47)
    a = run_gpu(w, x, out="bf16", grad="bf16")
    b = run_gpu(w, x, out="bf16", grad="bf16")
    for n in FIELDS:
        assert np.array_equal(a[n], b[n]), n
    ref = run_oracle(w, x)
    for n in ("o", "dq", "dk", "dv"):
        r = ref[n]
        half_ulp = np.abs(r) * 2.0 ** -9
        err = np.abs(a[n].astype(np.float64) - r)
        assert np.all(err <= half_ulp + tolerance(w, r)), n


@pytest.mark.parametrize("d", [64, 16])
def test_backward_reusing_the_forward_states_is_bit_identical(d):
    """DR_FLAG_REUSE_FWD: the chunk-start states the forward left give the same bits as
    the backward's own recomputation (both slice counts: d = 64 four slices, d = 16 one)."""
    w = inputs.small("gdn2", H=2, dk=d, dv=d, chunk=64, io="bf16", lengths=[100, 0, 64, 131])
    x = inputs.make_gdn2(w, seed=48)
    a = run_gpu(w, x, reuse=True)
    b = run_gpu(w, x, reuse=False)
    for n in FIELDS:
        assert np.array_equal(a[n], b[n]), n
