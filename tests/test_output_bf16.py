"""bf16-written o against the fp64 oracle, through the C ABI.

With a bf16 output the forward scan stages each whole chunk's o in shared memory and
writes it with tensor stores, and writes a ragged last chunk token by token.  The
cases cover one 128-row value tile per (sequence, head) (at least 120 units) and two
64-row tiles (fewer units), whole and ragged chunks, dense and packed sequences.  The
bound is the tolerance of tests/parity.py plus half a bf16 ulp of the value (the final
rounding of o to bf16).
"""
import numpy as np
import pytest

from delta_rule_recurrent_gated_gb300 import inputs

from parity import record, run_gpu, run_oracle, tolerance

pytestmark = pytest.mark.gpu

CASES = [
    ("gdn", dict(B=8, T=130, H=16)),     # 128 units: 128-row value tiles; chunks 64, 64, 2
    ("kda", dict(B=8, T=192, H=16)),     # 128 units, whole chunks only
    ("deltanet", dict(B=2, T=200, H=2)),  # 4 units: 64-row value tiles; a ragged tail
    ("gdn", dict(H=8, lengths=[64, 1, 130, 0, 63, 257] * 3)),  # packed, 144 units
]


@pytest.mark.parametrize("variant,shape", CASES)
def test_bf16_o_against_oracle(variant, shape):
    w = inputs.small(variant, dk=128, dv=128, **shape)
    x = inputs.make(w, seed=81)
    got = run_gpu(w, x, out="bf16", grad="bf16", backward=False)
    ref = run_oracle(w, x, backward=False)
    r = ref["o"]
    err = np.abs(got["o"].astype(np.float64) - r)
    tol = tolerance(w, r)
    record(w, "o (bf16)", float(err.max()) if err.size else 0.0, float(np.abs(r).max()) if r.size else 0.0, tol)
    assert np.all(np.isfinite(got["o"]))
    assert np.all(err <= np.abs(r) * 2.0 ** -9 + tol), float(err.max())
    # hT is written in fp32 either way
    assert float(np.max(np.abs(got["hT"] - ref["hT"]))) <= tolerance(w, ref["hT"])


# bf16 gradients (the step the benchmark times writes dq, dk, dv in bf16): each within the
# same bound, half a bf16 ulp of the value over the tolerance; dbeta, dg and dh0 are fp32
GRAD_CASES = [
    ("gdn", 128, dict(B=8, T=130, H=16)),      # 128-row value tiles, a ragged last chunk
    ("kda", 128, dict(B=2, T=200, H=2)),       # 64-row value tiles
    ("deltanet", 128, dict(H=2, lengths=[100, 0, 64, 1, 191, 7])),  # packed
    ("gdn", 64, dict(B=2, T=200, H=3)),        # d = 64: 64-channel rows per store
]


@pytest.mark.parametrize("variant,d,shape", GRAD_CASES)
def test_bf16_gradients_against_oracle(variant, d, shape):
    w = inputs.small(variant, dk=d, dv=d, **shape)
    x = inputs.make(w, seed=82)
    got = run_gpu(w, x, out="bf16", grad="bf16")
    ref = run_oracle(w, x)
    for name in ("dq", "dk", "dv", "dbeta", "dg", "dh0"):
        if ref.get(name) is None or got.get(name) is None:
            continue
        r = ref[name]
        g = got[name].astype(np.float64)
        assert np.all(np.isfinite(g)), name
        err = np.abs(g - r)
        tol = tolerance(w, r)
        record(w, f"{name} (bf16)", float(err.max()) if err.size else 0.0,
               float(np.abs(r).max()) if r.size else 0.0, tol)
        assert np.all(err <= np.abs(r) * 2.0 ** -9 + tol), (name, float(err.max()))
