"""GPU parity of the fp32 CUDA-core path against the fp64 oracle (tolerance
1e-4 max-abs), through the C ABI."""
import pytest

from delta_rule_recurrent_gated_gb300 import inputs

from parity import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def test_deltanet_f32_b1_t64_h2_d16():
    w = inputs.get("deltanet_f32_b1_t64_h2_d16")
    x = inputs.make(w, seed=0)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
@pytest.mark.parametrize("chunk,dk,dv", [(16, 16, 32), (32, 32, 32), (64, 64, 64), (16, 64, 16),
                                         (64, 128, 128), (16, 128, 128), (32, 128, 64),
                                         (64, 16, 128)])
def test_f32_small(variant, chunk, dk, dv):
    w = inputs.small(variant, B=2, T=150, H=2, dk=dk, dv=dv, chunk=chunk, io="f32")
    x = inputs.make(w, seed=1)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("variant", ["gdn", "kda"])
def test_f32_packed_ragged(variant):
    w = inputs.small(variant, H=2, dk=32, dv=32, chunk=16, io="f32", lengths=[37, 0, 16, 81, 1])
    x = inputs.make(w, seed=2)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


@pytest.mark.parametrize("variant", ["deltanet", "kda"])
def test_f32_d128_packed_ragged(variant):
    w = inputs.small(variant, H=2, dk=128, dv=128, chunk=64, io="f32",
                     lengths=[70, 0, 64, 129, 1])
    x = inputs.make(w, seed=3)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))
