"""Failure detection on the GPU without a GPU fault.

A kernel wait that runs out (an mbarrier nothing arrives on) must end with an
error code the host reads, and leave the context usable for the next call.
"""

import pytest
import torch

from block_diffusion_masked_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_masked_gb300 import binding, build

    build.build()
    binding.lib()
    return binding


def test_bounded_wait_reports_timeout_and_context_survives(b):
    assert b.dfa_status() == b.DFA_OK
    b.dfa_selftest_wait_timeout(20000)  # 20 ms
    assert b.dfa_status() == b.DFA_ETIMEOUT
    assert b.dfa_status() == b.DFA_OK  # read-and-clear
    # the context still runs real work
    q, k, v, _ = (t.cuda() for t in inputs.make_inputs(1, 64, 1, 64, seed=9))
    out, lse = b.dfa_forward(q, k, v, 4)
    torch.cuda.synchronize()
    assert b.dfa_status() == b.DFA_OK
    assert torch.isfinite(out.float()).all()


def test_selftest_argument_checks(b):
    with pytest.raises(b.DfaError):
        b.dfa_selftest_wait_timeout(0)
    with pytest.raises(b.DfaError):
        b.dfa_selftest_wait_timeout(2_000_000)
