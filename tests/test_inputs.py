"""The seeded synthetic inputs (delta_rule_recurrent_gated_gb300/inputs.py) follow their
stated recipes: shapes and dtypes, unit-norm q / k rows, beta in (0, 1), log-gates
<= 0, gate shapes per variant, ragged lengths, and determinism by seed."""
import numpy as np
import pytest
import torch

from delta_rule_recurrent_gated_gb300 import inputs


@pytest.mark.parametrize("variant", ["deltanet", "gdn", "kda"])
def test_prepared_inputs_recipe(variant):
    w = inputs.small(variant, B=2, T=70, H=3, dk=64, dv=32)
    x = inputs.make(w, seed=5)
    assert x["q"].shape == (2, 70, 3, 64) and x["v"].shape == (2, 70, 3, 32)
    assert x["q"].dtype == torch.bfloat16 and x["beta"].dtype == torch.float32
    norms = x["q"].float().norm(dim=-1)
    assert torch.all((norms - 1).abs() < 2e-2)  # unit rows, rounded to bf16
    assert torch.all((x["beta"] > 0) & (x["beta"] < 1))
    if variant == "deltanet":
        assert x["g"] is None
    else:
        shape = (2, 70, 3) if variant == "gdn" else (2, 70, 3, 64)
        assert x["g"].shape == shape and torch.all(x["g"] <= 0)
        # -softplus(N(0,1)) * 0.1: between -0.1 * softplus(6) and 0
        assert torch.all(x["g"] > -0.61)
    assert x["h0"].shape == (2, 3, 64, 32) and x["dhT"].shape == (2, 3, 64, 32)


def test_seeds_are_deterministic_and_distinct():
    w = inputs.small("kda", B=1, T=20, H=2, dk=16, dv=16, io="f32")
    a, b, c = inputs.make(w, seed=3), inputs.make(w, seed=3), inputs.make(w, seed=4)
    for n in ("q", "k", "v", "beta", "g", "h0", "dO", "dhT"):
        assert torch.equal(a[n], b[n]), n
    assert not torch.equal(a["q"], c["q"])


def test_ragged_lengths():
    lens = inputs.ragged_lengths(32768, 256, 4096, seed=0)
    assert sum(lens) == 32768
    assert all(256 <= L <= 4096 for L in lens[:-1]) and 1 <= lens[-1] <= 4096
    assert lens == inputs.ragged_lengths(32768, 256, 4096, seed=0)
    w = inputs.get("gdn_varlen_t32768_h16_d128")
    cu = inputs.cu_seqlens_of(w)
    assert cu[0] == 0 and cu[-1] == 32768 and torch.all(cu[1:] >= cu[:-1])
    assert inputs.num_seqs(w) == len(lens)


def test_explicit_lengths_with_empty_sequence():
    w = inputs.small("gdn", H=2, dk=16, dv=16, lengths=[5, 0, 3])
    x = inputs.make(w, seed=1)
    assert w.B == 1 and w.T == 8 and x["N"] == 3
    assert x["cu_seqlens"].tolist() == [0, 5, 5, 8]
    assert x["h0"].shape[0] == 3


def test_raw_inputs_recipe():
    w = inputs.small("kda", B=2, T=40, H=2, dk=64, dv=64)
    x = inputs.make_raw(w, seed=2)
    norms = x["q"].float().norm(dim=-1)
    assert norms.mean() > 4  # N(0,1) rows of 64 values, not normalised
    g = -torch.nn.functional.softplus(x["g"])  # the gate the library will form
    assert abs(float(g.mean()) + 0.806) < 0.1  # E softplus(N(0,1)) = 0.806
    assert x["beta"].min() < 0 < x["beta"].max()  # logits, not probabilities


def test_gdn2_inputs_recipe():
    w = inputs.get("gdn2_b4_t2048_h8_d64")
    x = inputs.make_gdn2(inputs.replace(w, T=64), seed=0)
    assert x["erase"].shape == (4, 64, 8, 64) and x["write"].shape == (4, 64, 8, 64)
    for n in ("erase", "write"):
        assert torch.all((x[n] > 0) & (x[n] < 1))
    assert x["g"].shape == (4, 64, 8) and torch.all(x["g"] <= 0)
    assert np.allclose(x["q"].float().norm(dim=-1).numpy(), 1, atol=2e-2)
