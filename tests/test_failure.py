"""The device failure path, tested without faulting the GPU: every tensor-core
kernel waits on mbarriers with a bounded wait and records DR_ERR_TIMEOUT in the
workspace error word when one runs out.  dr_selftest_wait runs that wait on a
barrier phase nothing completes (a flag that nothing sets), with a 1 ms limit; the
status must read DR_ERR_TIMEOUT, the context must stay usable (a full forward and
backward right after is correct and reports DR_OK), and the same wait on a phase
that does complete must report DR_OK."""
import pytest
import torch

from delta_rule_recurrent_gated_gb300 import binding, inputs

from parity import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_expired_wait_is_reported_and_the_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert binding.selftest_wait(ws.data_ptr(), False, 1_000_000, _stream()) == binding.DR_OK
    assert binding.check_status(ws.data_ptr(), _stream()) == binding.DR_ERR_TIMEOUT
    # the GPU and this context still work: a whole step, checked against the oracle
    w = inputs.small("gdn", B=2, T=130, H=2, dk=64, dv=64)
    x = inputs.make(w, seed=51)
    compare(w, x, run_gpu(w, x), run_oracle(w, x))


def test_completed_wait_reports_ok():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ws[:4] = 7  # stale word: the call clears it first
    assert binding.selftest_wait(ws.data_ptr(), True, 1_000_000, _stream()) == binding.DR_OK
    assert binding.check_status(ws.data_ptr(), _stream()) == binding.DR_OK


def test_a_problem_after_a_timeout_starts_clean():
    """The forward clears the error word it reports through, so a timeout recorded by an
    earlier call on the same workspace does not leak into a later one."""
    w = inputs.small("kda", B=1, T=70, H=2, dk=64, dv=64)
    x = inputs.make(w, seed=52)
    prob = binding.Problem(w.variant, w.B, w.T, w.H, w.dk, w.dv, device="cuda")
    assert binding.selftest_wait(prob.ws.data_ptr(), False, 100_000, _stream()) == binding.DR_OK
    assert prob.status() == binding.DR_ERR_TIMEOUT
    run_gpu(w, x, prob=prob)  # asserts DR_OK after the step
