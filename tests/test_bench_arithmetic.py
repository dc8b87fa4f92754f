"""The roofline arithmetic of bench.py, checked on the CPU against figures worked out
independently: the whole path's FLOPs and bytes per token and head at d = 128
(693,589 FLOPs; DeltaNet 2,828 B, Gated DeltaNet 2,840 B, KDA 4,364 B), the
design bytes of each kernel launch, the fp32 peak from unit counts and clock, and
the Gated DeltaNet-2 FLOP count restated from its product list, and each kernel's
share of the path's bytes."""
import importlib.util
import os

import pytest

from delta_rule_recurrent_gated_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("variant,bytes_per", [("deltanet", 2828), ("gdn", 2840),
                                               ("kda", 4364)])
def test_path_flops_and_bytes_per_token_head(bench, variant, bytes_per):
    w = inputs.Workload("t", variant, 1, 4096, 1, 128, 128)
    flops, byts = bench.algorithmic(w, 1)
    # F = 24 C d + 14 C d + 22 d^2 + 16/3 C^2 at C = 64, d = 128
    assert flops / 4096 == pytest.approx(24 * 64 * 128 + 14 * 64 * 128 + 22 * 128 * 128
                                         + 16 / 3 * 64 * 64)
    assert round(flops / 4096) == 693589
    assert byts / 4096 == bytes_per


def test_headline_state_bytes(bench):
    w = inputs.get("gdn_h0_b8_t4096_h16_d128")
    _, with_state = bench.algorithmic(w, 8)
    _, without = bench.algorithmic(inputs.replace(w, h0=False), 8)
    # h0 read by the forward and again by the backward, hT written, dhT read, dh0 written
    assert with_state - without == 5 * 128 * 128 * 4 * 8 * 16


def test_kernel_design_bytes(bench):
    w = inputs.get("gdn_h0_b8_t4096_h16_d128")
    th, recs = 8 * 4096 * 16, 8 * 64 * 16
    tile, dd = 64 * 128 * 2, 128 * 128 * 2
    assert bench.kernel_bytes("tc_prep", w, 8) == th * (3 * 256 + 4 + 4) + recs * (5 * tile + 8192 + 512)
    assert bench.kernel_bytes("tc_bwd_chunk", w, 8) == (
        th * (8 * 128 + 8) + recs * (2 * tile + 2 * dd + 8192 + 512) + th * (6 * 128 + 8))
    # the recorded capture of this workload, while the kernel source is the captured one
    t = bench.measured_traffic("tc_bwd_chunk", w)
    assert t is None or t == 1418410240 + 383005184
    assert bench.measured_traffic("tc_bwd_chunk", inputs.get("gdn_b2_t4096_h16_d128")) is None


def test_fp32_peak_and_gdn2_flops(bench):
    assert bench.fp32_alu_peak_tflops(2070) == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
    C = d = 64
    fwd = 2 * (11 * C * C * d) + C ** 3 / 3 + 2 * (4 * C * d * d)
    bwd = 2 * (20 * C * C * d) + 2 * (8 * C * d * d) + 2 * (2 * C ** 3)
    assert bench.gdn2_flops_per_chunk(C, d) == pytest.approx(fwd + bwd)


@pytest.mark.parametrize("name", ["gdn_h0_b8_t4096_h16_d128", "kda_b8_t4096_h16_d128",
                                  "sweep_deltanet_b16_t4096_h16_d128", "gdn_b4_t2048_h8_d64"])
def test_kernel_shares_add_up_to_the_path_bytes(bench, name):
    """Each kernel's share of the algorithmic bytes (what bench.py divides by the
    kernel's own time) sums to the whole path's algorithmic bytes."""
    w = inputs.get(name)
    N = w.B
    _, byts = bench.algorithmic(w, N)
    parts = sum(bench.kernel_algorithmic_bytes(k, w, N)
                for k in ("tc_prep", "tc_scan_fwd", "tc_scan_bwd", "tc_bwd_chunk"))
    assert parts == byts
    # tc_bwd_chunk of the headline: q, k, v, dO in; dq, dk, dv out (bf16); beta, g, dbeta, dg
    if name == "gdn_h0_b8_t4096_h16_d128":
        assert bench.kernel_algorithmic_bytes("tc_bwd_chunk", w, N) == 8 * 4096 * 16 * 1808


def test_both_arms_share_the_config(bench):
    w = inputs.get("gdn_h0_b8_t4096_h16_d128")
    c = bench.config_of(w, 1)
    assert c["chunk"] == 64 and c["seq_len"] == 4096 and c["heads"] == 16 and c["d_k"] == 128
