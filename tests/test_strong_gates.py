"""GPU parity under strong decay gates, through the C ABI, against the fp64 oracle.

The specified workloads draw log-gates g = -softplus(N(0,1)) * 0.1, about -0.08 per
token.  A layer may produce much stronger ones: the plain map of the projection,
-softplus(N(0,1)) (about -0.8 per token, a 64-token chunk decaying by about e^-50
per key channel), or twice that, where a chunk's cumulative log-decay passes -100
(e^-100 is below the fp32 range, so no factor e^{+-Gamma} taken from the chunk's
first token can be formed).  Every output and gradient must stay finite and within
the tolerance of tests/parity.py, for KDA (per key channel) and Gated DeltaNet
(per token), forward and backward, dense and packed.
"""
import numpy as np
import pytest

from delta_rule_recurrent_gated_gb300 import inputs

from parity import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def chunk_log_decay_min(w, x):
    """Most negative cumulative log-decay over any chunk and key channel."""
    g = x["g"].double().numpy()
    if w.variant == "gdn":
        g = g[..., None]
    worst = 0.0
    for t0 in range(0, w.T, w.chunk):
        worst = min(worst, float(g[:, t0:t0 + w.chunk].sum(axis=1).min()))
    return worst


@pytest.mark.parametrize("variant", ["kda", "gdn"])
@pytest.mark.parametrize("gate_scale,d", [(1.0, 128), (1.0, 64), (2.0, 128), (2.0, 64)])
def test_strong_gates_fwd_bwd(variant, gate_scale, d):
    w = inputs.replace(inputs.small(variant, B=2, T=200, H=2, dk=d, dv=d), gate_scale=gate_scale)
    x = inputs.make(w, seed=71)
    if gate_scale == 2.0:
        assert chunk_log_decay_min(w, x) < -100.0  # the case the chunk-start reference cannot take
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("variant", ["kda", "gdn"])
def test_strong_gates_packed(variant):
    w = inputs.replace(inputs.small(variant, H=2, dk=128, dv=128, lengths=[100, 0, 64, 1, 191, 7]),
                       gate_scale=2.0)
    x = inputs.make(w, seed=72)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


def test_strong_gates_full_size_kda():
    """KDA at its full workload size with the plain -softplus gates: every head of one
    sampled sequence against the oracle."""
    from test_parity_full import check_sampled, pick
    w = inputs.replace(inputs.get("kda_b8_t4096_h16_d128"), gate_scale=1.0)
    x = inputs.make(w, seed=73)
    got = run_gpu(w, x, reuse=True)
    check_sampled(w, x, got, pick(w, x, 1, seed=3))
    assert np.all(np.isfinite(got["o"]))


@pytest.mark.parametrize("variant", ["kda", "gdn"])
@pytest.mark.parametrize("chunk,d", [(64, 64), (64, 128), (32, 32)])
def test_strong_gates_fp32_path(variant, chunk, d):
    """The fp32 CUDA-core path under the same gates, at its 1e-4 bound."""
    w = inputs.replace(inputs.small(variant, B=2, T=150, H=2, dk=d, dv=d, chunk=chunk, io="f32"),
                       gate_scale=2.0)
    x = inputs.make(w, seed=74)
    if chunk == 64:
        assert chunk_log_decay_min(w, x) < -100.0
    compare(w, x, run_gpu(w, x), run_oracle(w, x))
