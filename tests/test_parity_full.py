"""GPU parity at the full workload sizes, in the launch configuration bench.py
times (bf16 io), on sampled (sequence, head) units that the fp64 oracle
computes one by one: the GPU runs the whole batch, the oracle reruns the
sampled sequences alone (same values, state carried from their own h0) and
every output and gradient of those units is compared element by element.
Tolerance: tests/parity.py (fp32-written outputs)."""
import numpy as np
import pytest
import torch

import oracle
from delta_rule_recurrent_gated_gb300 import inputs

from parity import check, run_gpu

pytestmark = pytest.mark.gpu


def oracle_for_sequence(w, x, n, heads):
    """Oracle outputs of sequence n, heads `heads`, as a one-sequence problem."""
    cu = x["cu_seqlens"]
    if cu is None:
        sl = (slice(n, n + 1), slice(None))
    else:
        sl = (slice(0, 1), slice(int(cu[n]), int(cu[n + 1])))

    def cut(t):
        return None if t is None else t[sl[0], sl[1]]

    def st(t):
        return None if t is None else t[n:n + 1]

    a = dict(q=cut(x["q"]), k=cut(x["k"]), v=cut(x["v"]), beta=cut(x["beta"]),
             g=cut(x["g"]), h0=st(x["h0"]), scale=w.scale,
             units=np.array(heads, dtype=np.int32))
    o, hT = oracle.forward(w.variant, **a)
    g = oracle.backward(w.variant, dO=cut(x["dO"]), dhT=st(x["dhT"]), **a)
    return sl, dict(o=o, hT=hT, **g)


def check_sampled(w, x, got, samples):
    worst = {}
    for n, heads in samples:
        sl, ref = oracle_for_sequence(w, x, n, heads)
        for name, r in ref.items():
            if r is None or got.get(name) is None:
                continue
            if name in ("hT", "dh0"):
                gsel = got[name][n:n + 1]
            else:
                gsel = got[name][sl[0], sl[1]]
            for h in heads:
                rr = r[:, h] if name in ("hT", "dh0") else r[:, :, h]
                gg = gsel[:, h] if name in ("hT", "dh0") else gsel[:, :, h]
                err, tol = check(w, name, gg, rr)
                worst[name] = max(worst.get(name, 0.0), err / tol)
                assert err <= tol, f"{w.name} seq {n} head {h} {name}: err {err} > tol {tol}"
    return worst


def pick(w, x, count, seed=0):
    """`count` sequences drawn without replacement (plus the shortest and the
    longest of a packed batch), each with all of its heads."""
    rng = np.random.default_rng(seed)
    N = x["N"]
    seqs = sorted(set(int(s) for s in rng.choice(N, size=min(count, N), replace=False)))
    if x["cu_seqlens"] is not None:
        lens = np.diff(x["cu_seqlens"].numpy())
        seqs = sorted(set(seqs) | {int(np.argmin(lens)), int(np.argmax(lens))})
    return [(n, list(range(w.H))) for n in seqs]


@pytest.mark.parametrize("name,count", [
    ("gdn_b4_t2048_h8_d64", 4),
    ("kda_b8_t4096_h16_d128", 3),
    ("gdn_h0_b8_t4096_h16_d128", 3),
    ("gdn_varlen_t32768_h16_d128", 3),
    ("sweep_deltanet_b16_t4096_h16_d128", 2),
    ("sweep_gdn_b4_t16384_h16_d128", 1),
    ("sweep_kda_b8_t8192_h16_d128", 1),
    ("sweep_gdn_b8_t8192_h16_d128", 1),
    ("sweep_kda_b4_t16384_h16_d128", 1),
    ("sweep_deltanet_b2_t32768_h16_d128", 1),
    ("sweep_gdn_b2_t32768_h16_d128", 1),
    ("sweep_kda_b2_t32768_h16_d128", 1),
])
def test_full_size_sampled(name, count):
    w = inputs.get(name)
    x = inputs.make(w, seed=0)
    got = run_gpu(w, x, reuse=True)
    check_sampled(w, x, got, pick(w, x, count))
    torch.cuda.empty_cache()


def test_determinism_full_size():
    """Two runs of the same call give bit-identical outputs and gradients."""
    w = inputs.get("kda_b8_t4096_h16_d128")
    x = inputs.make(w, seed=1)
    a = run_gpu(w, x, reuse=True, out="bf16", grad="bf16")
    b = run_gpu(w, x, reuse=True, out="bf16", grad="bf16")
    for n in ("o", "hT", "dq", "dk", "dv", "dbeta", "dg", "dh0"):
        assert np.array_equal(a[n], b[n]), n
