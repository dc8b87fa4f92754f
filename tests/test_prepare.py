"""GPU parity of the input-preparation mode (DR_FLAG_PREPARE_INPUTS) against the
fp64 oracle (oracle/prepare.py composed with the recurrence), through the C ABI:
raw q, k (not normalised), beta logits and gate arguments go in; o, hT and the
gradients with respect to the raw tensors come out.  Covers both paths (bf16
tensor cores, fp32 CUDA cores), ragged tails, packed sequences, zero q / k rows
(the eps of the normalisation), the emitted write and its gradient, the
recurrent step, and the full workload sizes on sampled (sequence, head) units.
Tolerance: tests/parity.py."""
import numpy as np
import pytest
import torch

from oracle import prepare as prep
from delta_rule_recurrent_gated_gb300 import binding, inputs

from parity import check, compare, run_gpu, tolerance

pytestmark = pytest.mark.gpu

VARIANTS = ["deltanet", "gdn", "kda"]


def problem(w, x, out="f32", grad="f32"):
    return binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io=w.io,
                           out=out, grad=grad, scale=w.scale, cu_seqlens=x["cu_seqlens"],
                           device="cuda", prepare=True)


def oracle_raw(w, x, units=None, backward=True):
    a = dict(scale=w.scale, cu_seqlens=x["cu_seqlens"], units=units)
    o, hT = prep.forward_raw(w.variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], **a)
    res = {"o": o, "hT": hT}
    if backward:
        res.update(prep.backward_raw(w.variant, x["q"], x["k"], x["v"], x["beta"], x["g"],
                                     x["h0"], x["dO"], x["dhT"], **a))
    return res


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("io,d,chunk", [("bf16", 128, 64), ("bf16", 64, 64), ("f32", 32, 16),
                                        ("f32", 64, 64)])
def test_prepared_fwd_bwd_small(variant, io, d, chunk):
    w = inputs.small(variant, B=2, T=200, H=3, dk=d, dv=d, chunk=chunk, io=io)
    x = inputs.make_raw(w, seed=31)
    compare(w, x, run_gpu(w, x, prob=problem(w, x)), oracle_raw(w, x))


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_prepared_packed(variant):
    w = inputs.small(variant, H=2, dk=128, dv=128, lengths=[100, 0, 64, 1, 191, 7])
    x = inputs.make_raw(w, seed=32)
    compare(w, x, run_gpu(w, x, prob=problem(w, x)), oracle_raw(w, x))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("d", [64, 128])
def test_prepared_zero_rows(variant, d):
    """A zero q or k row maps to the zero vector (eps keeps the scale finite); its
    raw gradient is the prepared one times 1/sqrt(eps) = 1000.  bf16 io only: the
    fp32 bar of 1e-4 absolute is below fp32 rounding of a gradient amplified a
    thousandfold."""
    w = inputs.small(variant, B=2, T=70, H=2, dk=d, dv=d)
    x = inputs.make_raw(w, seed=33)
    x["q"][0, 5, 1] = 0
    x["q"][1, 69, 0] = 0
    x["k"][1, 40, 1] = 0
    x["k"][0, 0, 0] = 0
    compare(w, x, run_gpu(w, x, prob=problem(w, x)), oracle_raw(w, x))


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_prepared_reuse_matches_recompute(variant):
    w = inputs.small(variant, B=2, T=300, H=2, dk=128, dv=128)
    x = inputs.make_raw(w, seed=34)
    prob = problem(w, x)
    a = run_gpu(w, x, prob=prob, reuse=True)
    b = run_gpu(w, x, prob=prob, reuse=False)
    for n in ("o", "hT", "dq", "dk", "dv", "dbeta", "dg", "dh0"):
        assert np.array_equal(a[n], b[n]), n


@pytest.mark.parametrize("variant", VARIANTS)
def test_prepared_write_and_its_gradient(variant):
    w = inputs.small(variant, B=2, T=150, H=2, dk=64, dv=64)
    x = inputs.make_raw(w, seed=35)
    dU = torch.randn(x["v"].shape, generator=torch.Generator().manual_seed(5)).to(x["v"].dtype)
    prob = problem(w, x)
    t = {n: (v.cuda() if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    u = torch.empty(w.B, w.T, w.H, w.dv, dtype=torch.float32, device="cuda")
    o, hT = prob.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], u=u)
    gr = prob.backward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"], t["dO"], t["dhT"],
                       reuse_fwd=True, dU=dU.cuda())
    torch.cuda.synchronize()
    assert prob.status() == binding.DR_OK
    got = {"o": o, "hT": hT, "u": u, **gr}
    got = {n: (None if v is None else v.float().cpu().numpy()) for n, v in got.items()}
    a = dict(scale=w.scale)
    ro, rh, ru = prep.forward_raw(w.variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                                  want_u=True, **a)
    ref = {"o": ro, "hT": rh, "u": ru}
    ref.update(prep.backward_raw(w.variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                                 x["dO"], x["dhT"], dU=dU, **a))
    compare(w, x, got, ref, fields=("o", "hT", "u", "dq", "dk", "dv", "dbeta", "dg", "dh0"))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("io,d", [("bf16", 128), ("f32", 64), ("f32", 16)])
def test_prepared_decode_matches_the_recurrence(variant, io, d):
    """dr_decode with the flag: token-by-token calls on raw inputs reproduce the
    oracle's prepared forward (outputs of every token and the final state)."""
    w = inputs.replace(inputs.small(variant, B=3, T=9, H=2, dk=d, dv=d, io=io), scale=0.5)
    x = inputs.make_raw(w, seed=36, need_grad_inputs=False)
    o_ref, h_ref = prep.forward_raw(w.variant, x["q"], x["k"], x["v"], x["beta"], x["g"],
                                    x["h0"], scale=w.scale)
    dev = torch.device("cuda:0")
    dec = binding.Decoder(variant, w.B, 1, w.H, d, d, io=io, out="f32", scale=w.scale,
                          device=dev, prepare=True)
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
    for name, got, ref in (("o", o, o_ref), ("state", state.cpu().numpy(), h_ref)):
        err, tol = check(w, name, got, ref)
        assert err <= tol, f"{w.name} {name}: err {err}"


def _oracle_unit(w, x, n, h):
    """Oracle outputs of sequence n, head h, as a one-sequence, one-head problem."""
    cu = x["cu_seqlens"]
    rows = slice(n, n + 1) if cu is None else slice(0, 1)
    toks = slice(None) if cu is None else slice(int(cu[n]), int(cu[n + 1]))

    def cut(t):
        return None if t is None else t[rows, toks, h:h + 1]

    def st(t):
        return None if t is None else t[n:n + 1, h:h + 1]

    a = dict(scale=w.scale)
    o, hT = prep.forward_raw(w.variant, cut(x["q"]), cut(x["k"]), cut(x["v"]), cut(x["beta"]),
                             cut(x["g"]), st(x["h0"]), **a)
    g = prep.backward_raw(w.variant, cut(x["q"]), cut(x["k"]), cut(x["v"]), cut(x["beta"]),
                          cut(x["g"]), st(x["h0"]), cut(x["dO"]), st(x["dhT"]), **a)
    return (rows, toks), dict(o=o, hT=hT, **g)


@pytest.mark.parametrize("name", ["gdn_h0_b8_t4096_h16_d128", "kda_b8_t4096_h16_d128"])
def test_prepared_full_size_sampled(name):
    w = inputs.get(name)
    x = inputs.make_raw(w, seed=0)
    got = run_gpu(w, x, prob=problem(w, x), reuse=True)
    rng = np.random.default_rng(1)
    for n in sorted(set(int(s) for s in rng.choice(x["N"], size=2, replace=False))):
        h = int(rng.integers(w.H))
        (rows, toks), ref = _oracle_unit(w, x, n, h)
        for fname, r in ref.items():
            if r is None or got.get(fname) is None:
                continue
            if fname in ("hT", "dh0"):
                gg = got[fname][n:n + 1, h:h + 1]
            else:
                gg = got[fname][rows, toks, h:h + 1]
            err, tol = check(w, fname, gg, r)
            assert err <= tol, f"{name} seq {n} head {h} {fname}: err {err} > tol {tol}"
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_prepared_bf16_outputs_and_gradients(variant):
    """bf16-written o and gradients (the bench's precision) in the preparation mode,
    against the oracle within half a bf16 ulp on top of the tolerance."""
    w = inputs.small(variant, B=2, T=150, H=2, dk=128, dv=128)
    x = inputs.make_raw(w, seed=37)
    got = run_gpu(w, x, prob=problem(w, x, out="bf16", grad="bf16"))
    ref = oracle_raw(w, x)
    for n in ("o", "dq", "dk", "dv"):
        r = ref[n]
        err = np.abs(got[n].astype(np.float64) - r)
        assert np.all(err <= np.abs(r) * 2.0 ** -9 + tolerance(w, r)), n
