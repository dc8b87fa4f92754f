"""The no-allocation forward (dr_fwd_noalloc) against the regular dr_fwd.

dr_fwd_noalloc is for callers that cannot call cudaMalloc where they run the
layer (they are handed only input and output buffers, or an allocation there
is not allowed); its scratch is a static array inside the library rather than
a caller workspace.  This test calls it through the C ABI twice in a row, on
different inputs, and checks each result against dr_fwd on the same inputs
with the fp32 tolerance of the parity tests (1e-4 max-abs).  A problem larger
than the static scratch must be refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

from delta_rule_recurrent_gated_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else t.data_ptr()


def test_noalloc_forward_matches_dr_fwd_on_two_calls():
    lib = binding.load()
    dev = torch.device("cuda:0")
    w = inputs.small("kda", B=2, T=150, H=3, dk=32, dv=32, chunk=16, io="f32")
    stream = torch.cuda.current_stream(dev).cuda_stream
    for seed in (11, 12):
        x = inputs.make(w, seed=seed, need_grad_inputs=False)
        t = {n: (v.to(dev) if torch.is_tensor(v) else v) for n, v in x.items()}
        prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, chunk=w.chunk, io="f32",
                               out="f32", grad="f32", device=dev)
        o_ref, h_ref = prob.forward(t["q"], t["k"], t["v"], t["beta"], t["g"], t["h0"])
        o = torch.full_like(o_ref, float("nan"))
        hT = torch.full_like(h_ref, float("nan"))
        rc = lib.dr_fwd_noalloc(ctypes.byref(prob.desc), _ptr(t["q"]), _ptr(t["k"]),
                                _ptr(t["v"]), _ptr(t["beta"]), _ptr(t["g"]), _ptr(t["h0"]),
                                _ptr(o), _ptr(hT), stream)
        assert rc == binding.DR_OK, binding.error_string(rc)
        torch.cuda.synchronize(dev)
        for got, ref in ((o, o_ref), (hT, h_ref)):
            g = got.double().cpu().numpy()
            assert np.all(np.isfinite(g))
            assert float(np.max(np.abs(g - ref.double().cpu().numpy()))) <= 1e-4


def test_noalloc_refuses_problems_beyond_its_scratch():
    lib = binding.load()
    d = binding.DrDesc()
    d.B, d.T, d.H, d.d_k, d.d_v, d.chunk = 4, 64, 16, 32, 32, 16   # 64 (sequence, head) units
    d.variant, d.io_dtype, d.out_dtype, d.grad_dtype = binding.DR_GDN, binding.DR_F32, \
        binding.DR_F32, binding.DR_F32
    d.scale, d.flags, d.num_seqs = 1.0, 0, 4
    rc = lib.dr_fwd_noalloc(ctypes.byref(d), 16, 16, 16, 16, 16, None, 16, None, None)
    assert rc == binding.DR_ERR_SCRATCH_LIMIT
    assert "static scratch" in binding.error_string(rc)
    d.io_dtype = binding.DR_BF16
    d.d_k = d.d_v = 128
    d.chunk = 64
    rc = lib.dr_fwd_noalloc(ctypes.byref(d), 16, 16, 16, 16, 16, None, 16, None, None)
    assert rc == binding.DR_ERR_UNSUPPORTED
