"""GPU parity of the bf16 tensor-core path against the fp64 oracle, through the
C ABI, at sizes the oracle finishes in seconds (several chunks, ragged tails,
packed sequences, empty sequences) and at the full workload sizes on sampled
(sequence, head) units.  Tolerance: tests/parity.py."""
import numpy as np
import pytest

from delta_rule_recurrent_gated_gb300 import inputs

from parity import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

VARIANTS = ["deltanet", "gdn", "kda"]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("d", [64, 128])
def test_forward_small(variant, d):
    w = inputs.small(variant, B=2, T=200, H=3, dk=d, dv=d)
    x = inputs.make(w, seed=3)
    compare(w, x, run_gpu(w, x, backward=False), run_oracle(w, x, backward=False))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("T", [1, 63, 64, 65])
def test_forward_short_sequences(variant, T):
    w = inputs.small(variant, B=3, T=T, H=2, dk=64, dv=64)
    x = inputs.make(w, seed=4)
    compare(w, x, run_gpu(w, x, backward=False), run_oracle(w, x, backward=False))


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_forward_packed(variant):
    w = inputs.small(variant, H=2, dk=128, dv=128, lengths=[100, 0, 64, 1, 191, 7])
    x = inputs.make(w, seed=5)
    compare(w, x, run_gpu(w, x, backward=False), run_oracle(w, x, backward=False))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_bwd_small(variant, d):
    w = inputs.small(variant, B=2, T=200, H=3, dk=d, dv=d)
    x = inputs.make(w, seed=6)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("T", [1, 64, 130])
def test_fwd_bwd_short_and_tail(variant, T):
    w = inputs.small(variant, B=2, T=T, H=2, dk=64, dv=64, h0=False, dhT=False)
    x = inputs.make(w, seed=7)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("variant", VARIANTS)
def test_fwd_bwd_packed(variant):
    w = inputs.small(variant, H=2, dk=128, dv=128, lengths=[100, 0, 64, 1, 191, 7])
    x = inputs.make(w, seed=8)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


# 128 (sequence, head) units or more: the scans take 128-row value tiles, the shape of the
# full-size workloads, here with ragged tails and packed sequences at a size the oracle
# runs whole
@pytest.mark.parametrize("variant", VARIANTS)
def test_fwd_bwd_many_units_ragged(variant):
    w = inputs.small(variant, B=8, T=130, H=16, dk=128, dv=128)
    x = inputs.make(w, seed=11)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_fwd_bwd_many_units_packed(variant):
    w = inputs.small(variant, H=16, dk=128, dv=128, lengths=[200, 64, 1, 130, 0, 65, 191, 7])
    x = inputs.make(w, seed=12)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_backward_recompute_matches_reuse(variant):
    w = inputs.small(variant, B=2, T=300, H=2, dk=128, dv=128)
    x = inputs.make(w, seed=9)
    a = run_gpu(w, x, reuse=True)
    b = run_gpu(w, x, reuse=False)
    for n in ("dq", "dk", "dv", "dbeta", "dg", "dh0"):
        assert np.array_equal(a[n], b[n]), n


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("io,d,chunk", [("bf16", 128, 64), ("f32", 32, 16)])
def test_fwd_bwd_read_scale(variant, io, d, chunk):
    w = inputs.replace(inputs.small(variant, B=2, T=150, H=2, dk=d, dv=d, chunk=chunk, io=io),
                       scale=0.375)
    x = inputs.make(w, seed=10)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))
