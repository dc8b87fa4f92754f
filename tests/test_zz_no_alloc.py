"""The no-allocation forward (dr_fwd_noalloc) against the regular dr_fwd and the
fp64 oracle.

dr_fwd_noalloc is for callers that cannot call cudaMalloc where they run the
layer (they are handed only input and output buffers, or an allocation there
is not allowed); its scratch is a static array inside the library rather than
a caller workspace.  These tests call it through the C ABI and check its o and
hT against dr_fwd on the same inputs and against the oracle, with the fp32
tolerance of the parity tests (1e-4 max-abs): twice in a row on different
inputs, at the largest problem its scratch holds (46 sequence-head units at
d <= 64, 11 at d = 128), and on packed ragged sequences (where the unit count
is sequences x heads, not B x heads).  One unit more than the scratch holds
must be refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from delta_rule_recurrent_gated_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _ptr(t):
    return None if t is None else t.data_ptr()


def _noalloc_vs_fwd_and_oracle(w, seed):
    lib = binding.load()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    x = inputs.make(w, seed=seed, need_grad_inputs=False)
    t = {n: (v.to(dev) if torch.is_tensor(v) and n != "cu_seqlens" else v) for n, v in x.items()}
    prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io="f32",
                           out="f32", grad="f32", cu_seqlens=x["cu_seqlens"], device=dev)
    o_ref, h_ref = prob.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
    o = torch.full_like(o_ref, float("nan"))
    hT = torch.full_like(h_ref, float("nan"))
    rc = lib.dr_fwd_noalloc(ctypes.byref(prob.desc), _ptr(t["q"]), _ptr(t["k"]), _ptr(t["v"]),
                            _ptr(t["beta"]), _ptr(t["g"]), _ptr(t["h0"]), _ptr(o), _ptr(hT),
                            stream)
    assert rc == binding.DR_OK, binding.error_string(rc)
    torch.cuda.synchronize(dev)
    ro, rh = oracle.forward(w.variant, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                            cu_seqlens=x["cu_seqlens"])
    for got, lib_ref, ora in ((o, o_ref, ro), (hT, h_ref, rh)):
        g = got.double().cpu().numpy()
        assert np.all(np.isfinite(g))
        assert float(np.max(np.abs(g - lib_ref.double().cpu().numpy()))) <= TOL
        assert float(np.max(np.abs(g - ora))) <= TOL


def test_noalloc_forward_matches_dr_fwd_on_two_calls():
    w = inputs.small("kda", B=2, T=150, H=3, dk=32, dv=32, chunk=16, io="f32")
    for seed in (11, 12):
        _noalloc_vs_fwd_and_oracle(w, seed)


@pytest.mark.parametrize("variant,B,H,d", [("gdn", 2, 23, 64), ("deltanet", 1, 11, 128)])
def test_noalloc_at_its_largest_problem(variant, B, H, d):
    """46 units at d = 64 and 11 at d = 128 are accepted and correct."""
    w = inputs.small(variant, B=B, T=100, H=H, dk=d, dv=d, chunk=32, io="f32")
    _noalloc_vs_fwd_and_oracle(w, 13)


def test_noalloc_packed_ragged():
    w = inputs.small("gdn", H=3, dk=64, dv=64, chunk=64, io="f32", lengths=[70, 0, 1, 129, 64])
    _noalloc_vs_fwd_and_oracle(w, 14)


def _desc(B, H, d, chunk=16, io=binding.DR_F32, num_seqs=None, packed=False):
    dd = binding.DrDesc()
    dd.B, dd.T, dd.H, dd.d_k, dd.d_v, dd.chunk = B, 64, H, d, d, chunk
    dd.variant, dd.io_dtype, dd.out_dtype, dd.grad_dtype = binding.DR_GDN, io, binding.DR_F32, \
        binding.DR_F32
    dd.scale, dd.flags = 1.0, 0
    dd.num_seqs = B if num_seqs is None else num_seqs
    if packed:  # never dereferenced: the call is refused before any launch
        dd.cu_seqlens, dd.chunk_offsets, dd.chunk_table, dd.num_chunks = 16, 16, 16, 4
    return dd


def _call(dd):
    return binding.load().dr_fwd_noalloc(ctypes.byref(dd), 16, 16, 16, 16, 16, None, 16, None,
                                         None)


def test_noalloc_refuses_one_unit_beyond_its_scratch():
    assert _call(_desc(1, 47, 32)) == binding.DR_ERR_SCRATCH_LIMIT          # 47 units, d <= 64
    assert _call(_desc(1, 12, 128, chunk=64)) == binding.DR_ERR_SCRATCH_LIMIT  # 12 units, d = 128
    # packed: the units are sequences x heads (47), not B x heads (1 x 1)
    assert _call(_desc(1, 1, 32, num_seqs=47, packed=True)) == binding.DR_ERR_SCRATCH_LIMIT
    assert "static scratch" in binding.error_string(binding.DR_ERR_SCRATCH_LIMIT)
    dd = _desc(4, 16, 128, chunk=64, io=binding.DR_BF16)
    assert _call(dd) == binding.DR_ERR_UNSUPPORTED
